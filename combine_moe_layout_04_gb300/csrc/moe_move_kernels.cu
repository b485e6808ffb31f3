// moe_move_kernels.cu -- dispatch-permute and combine-unpermute on sm_103a.
//
// Both are HBM-bound row moves ("Poor HybridEP performance on dual-node 16x
// B300 GPUs": dispatch_with_permute / combine_with_unpermute), so they are
// written for bytes in flight, not for arithmetic.
//
//  * register movers (the default dispatch, quantise-in-dispatch, the
//    expert-group combine, and every combine with more than 8 partners): one
//    warp per (unit, column span), every load of the span issued before any
//    is used, 256-bit loads and stores where rows and bases allow; the grid
//    holds several times the CTAs that fit at once, so CTAs turn over instead
//    of looping.  On GB300 this kept the DRAM write stream fuller than the
//    shared-memory pipelines for the dispatch (read 1, write k) and for the
//    group combine's fp32 chain.
//  * bulk pipelines (the flat and relay combines with at most 8 partners; the
//    dispatch and the group combine on request): the Blackwell bulk-copy
//    engine (cp.async.bulk, "TMA") moves the rows.  Each warp runs its own
//    pipeline of shared-memory stages guarded by mbarriers.  Combine gathers
//    the partner pieces of one unit into a stage and reduces it from shared
//    memory (combine_bulk_kernel; combine_packed_kernel packs several column
//    pieces per partner into a stage when a unit has few partners); dispatch
//    loads one source chunk and writes it to its partner rows with bulk
//    stores.  Every barrier wait has a wall-time limit; a kernel that gives
//    up records a fault bit, drains its own copies and returns.
//
// Which rows a unit touches is a route (below): the flat path pairs a token
// with its k receive rows; the two hops of the Mode 2 relay pair a token with
// its relay rows, and a relay row with the receive rows it feeds.
// A partner row outside its buffer is skipped (dispatch) or contributes
// nothing (combine), so a bad layout cannot write out of bounds.

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMoveThreads = 256;
constexpr int kMoveWarps = kMoveThreads / 32;
constexpr unsigned kAll = 0xffffffffu;

// How a combine carries an fp32 chain across launches through an fp32 row per
// unit (h floats): kAccFirst starts the sum from 0 and stores the chain,
// kAccMid adds to the stored chain (and skips units with no partner),
// kAccLast adds to it and writes the bf16 row; kAccNone is a plain combine.
constexpr int kAccNone = 0, kAccFirst = 1, kAccMid = 2, kAccLast = 3;

// ---- routes ------------------------------------------------------------------
//
// A mover walks units; unit u owns one row of its own (the row a dispatch
// reads, the row a combine writes: self_row) and up to 32 partner rows, one
// per lane (the rows a dispatch writes, the rows a combine sums, with their
// weights).  partner() is called by all 32 lanes of a warp with the same u;
// live is false for a u past the end, which yields no partners.
//
// The lookup has two halves so that a mover can run it one unit ahead:
// raw() issues the loads of unit u's partners without using their values,
// resolve() turns them into (row, weight) when they are needed.  partner()
// is the two in a row.  Routes whose lookup needs its own values at once
// (a relay row's token, a token's hosts) do it all in raw().

struct RawPartner {
    int row;    // partner row as loaded (-1: none)
    float w;    // its weight
    int key;    // route-specific: the slot's expert (GroupSlotRoute)
};

// Flat: unit = token t; lane j < k: receive row pos[t, j], gate weight w[t, j].
struct SlotRoute {
    const int32_t* pos;
    const float* w;  // NULL for dispatch
    int T, k;
    int rows;        // receive rows: T * k
    __device__ __forceinline__ long long units() const { return T; }
    __device__ __forceinline__ int self_row(long long u) const { return (int)u; }
    __device__ __forceinline__ RawPartner raw(long long u, bool live, int lane) const {
        RawPartner r{-1, 0.0f, 0};
        if (live && lane < k) {
            const size_t i = (size_t)u * k + lane;
            r.row = pos[i];
            if (w != nullptr) r.w = w[i];
        }
        return r;
    }
    __device__ __forceinline__ void resolve(const RawPartner& r, int& row, float& wt) const {
        row = (r.row < 0 || r.row >= rows) ? -1 : r.row;
        wt = r.w;
    }
    __device__ __forceinline__ void partner(long long u, bool live, int lane, int& row, float& wt) const {
        resolve(raw(u, live, lane), row, wt);
    }
};

// Relay hop between a token and its relay rows: unit = token t; lane i: the
// relay row of the i-th host (ascending) that t reaches, weight 1.  A token
// reaches at most min(k, H) hosts.
struct HostRoute {
    const int32_t* relay_pos;  // [T][H]
    int T, H;
    int rows;                  // relay buffer rows
    __device__ __forceinline__ long long units() const { return T; }
    __device__ __forceinline__ int self_row(long long u) const { return (int)u; }
    __device__ __forceinline__ void partner(long long u, bool live, int lane, int& row, float& wt) const {
        int lo = -1, hi = -1;  // hosts lane and lane + 32
        if (live) {
            const int32_t* rp = relay_pos + (size_t)u * H;
            if (lane < H) lo = rp[lane];
            if (lane + 32 < H) hi = rp[lane + 32];
            if (lo >= rows) lo = -1;
            if (hi >= rows) hi = -1;
        }
        const unsigned mlo = __ballot_sync(kAll, lo >= 0), mhi = __ballot_sync(kAll, hi >= 0);
        const int nlo = __popc(mlo), n = nlo + __popc(mhi);
        // lane i takes the i-th set bit of (mhi:mlo)
        unsigned m = lane < nlo ? mlo : mhi;
        const int skip = lane < nlo ? lane : lane - nlo;
        for (int i = 0; i < skip && lane < n; ++i) m &= m - 1;
        const int from = lane < n ? __ffs(m) - 1 : 0;
        const int vlo = __shfl_sync(kAll, lo, from), vhi = __shfl_sync(kAll, hi, from);
        row = lane < n ? (lane < nlo ? vlo : vhi) : -1;
        wt = row >= 0 ? 1.0f : 0.0f;
    }
    __device__ __forceinline__ RawPartner raw(long long u, bool live, int lane) const {
        RawPartner r{-1, 0.0f, 0};
        partner(u, live, lane, r.row, r.w);
        return r;
    }
    __device__ __forceinline__ void resolve(const RawPartner& r, int& row, float& wt) const {
        row = r.row;
        wt = r.w;
    }
};

// Grouped relay hop of combine: unit = token t; lane j < k: receive row
// pos[t, j] with weight w[t, j], and key(j) = slot_relay[t, j], the relay row
// (one per host the token reaches) whose partial sum slot j joins.
struct TokenRelayRoute {
    const int32_t* pos;
    const float* w;
    const int32_t* slot_relay;  // [T * k]
    int T, k;
    int rows;                   // receive rows: T * k
    int cap;                    // relay buffer rows
    __device__ __forceinline__ long long units() const { return T; }
    __device__ __forceinline__ int self_row(long long u) const { return (int)u; }
    __device__ __forceinline__ void partner(long long u, bool live, int lane, int& row, float& wt) const {
        row = -1;
        wt = 0.0f;
        if (live && lane < k) {
            const size_t i = (size_t)u * k + lane;
            row = pos[i];
            wt = w[i];
            if (row < 0 || row >= rows) row = -1;
        }
    }
    __device__ __forceinline__ int key(long long u, bool live, int lane) const {
        if (!live || lane >= k) return -1;
        const int r = slot_relay[(size_t)u * k + lane];
        return (r >= 0 && r < cap) ? r : -1;
    }
};

// One expert group of the flat path: unit = token t; lane j < k: receive row
// pos[t, j] with weight w[t, j] when expert ids[t, j] is in group g.  raw()
// loads the id, the row and the weight side by side (the row and weight of a
// slot outside the group are loaded too, and dropped by resolve()).
struct GroupSlotRoute {
    const int32_t* pos;
    const float* w;             // NULL for dispatch
    const int32_t* ids;
    const int32_t* group;       // [E]
    int g;
    int T, k, E;
    int rows;                   // receive rows: T * k
    __device__ __forceinline__ long long units() const { return T; }
    __device__ __forceinline__ int self_row(long long u) const { return (int)u; }
    __device__ __forceinline__ RawPartner raw(long long u, bool live, int lane) const {
        RawPartner r{-1, 0.0f, -1};
        if (live && lane < k) {
            const size_t i = (size_t)u * k + lane;
            r.key = ids[i];
            r.row = pos[i];
            if (w != nullptr) r.w = w[i];
        }
        return r;
    }
    __device__ __forceinline__ void resolve(const RawPartner& r, int& row, float& wt) const {
        const bool in = r.key >= 0 && r.key < E && __ldg(group + r.key) == g;
        row = (in && r.row >= 0 && r.row < rows) ? r.row : -1;
        wt = in ? r.w : 0.0f;
    }
    __device__ __forceinline__ void partner(long long u, bool live, int lane, int& row, float& wt) const {
        resolve(raw(u, live, lane), row, wt);
    }
};

// Relay hop between a relay row and the receive rows it feeds: unit = relay
// row r of token t = relay_src[r]; lane j < k: receive row pos[t, j] with
// weight w[t, j] when slot j is fed by r (slot_relay[t, j] == r).  The number
// of relay rows is read on the device.
struct RelaySlotRoute {
    const int32_t* relay_src;   // [cap]
    const int32_t* slot_relay;  // [T * k]
    const int32_t* pos;
    const float* w;             // NULL for dispatch
    const int32_t* n_relay;     // device word: relay rows in use
    int T, k;
    int rows;                   // receive rows: T * k
    int cap;                    // relay buffer rows
    __device__ __forceinline__ long long units() const {
        const int n = __ldg(n_relay);
        return n < 0 ? 0 : (n < cap ? n : cap);
    }
    __device__ __forceinline__ int self_row(long long u) const { return (int)u; }
    __device__ __forceinline__ void partner(long long u, bool live, int lane, int& row, float& wt) const {
        row = -1;
        wt = 0.0f;
        if (live && lane < k) {
            const int t = relay_src[u];
            if (t >= 0 && t < T) {
                const size_t i = (size_t)t * k + lane;
                if (slot_relay[i] == (int)u) {
                    row = pos[i];
                    if (w != nullptr) wt = w[i];
                    if (row < 0 || row >= rows) row = -1;
                }
            }
        }
    }
    __device__ __forceinline__ RawPartner raw(long long u, bool live, int lane) const {
        RawPartner r{-1, 0.0f, 0};
        partner(u, live, lane, r.row, r.w);
        return r;
    }
    __device__ __forceinline__ void resolve(const RawPartner& r, int& row, float& wt) const {
        row = r.row;
        wt = r.w;
    }
};

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

// Lane i < n takes the i-th partner (ascending lane order) of p / w; n partners.
__device__ __forceinline__ void compact_partners(int lane, int p, float w, int& cp, float& cw, int& n) {
    const unsigned m = __ballot_sync(kAll, p >= 0);
    n = __popc(m);
    unsigned mm = m;
    for (int i = 0; i < lane && i < n; ++i) mm &= mm - 1;  // lane-th partner
    const int from = lane < n ? __ffs(mm) - 1 : 0;
    cp = __shfl_sync(kAll, p, from);
    cw = __shfl_sync(kAll, w, from);
    if (lane >= n) {
        cp = -1;
        cw = 0.0f;
    }
}

// ---- vector chain combine ----------------------------------------------------
//
// One expert group's combine through registers: one warp per (token, span of
// 32 x kChainU runs of 8 columns), on a grid of several times the resident
// CTAs.  Lane L holds runs L, L + 32, ... of the span: their fp32 chain
// values (32-byte loads and stores) and, for each partner, the matching 16
// bytes of bf16 y.  The partners are compacted in ascending lane order and
// summed kChainKB at a time, every load of a round issued before any is used,
// so each chain value takes its fma steps in the route's partner order.  Any
// number of partners (k <= 32).  Two runs a lane and three partners a round,
// from a sweep on GB300 (G = 4 group combines at prefill-fp8, sum of the four):
// U, KB = 2, 3: 699 us (63 registers, four CTAs an SM); 2, 2: 706; 1, 1 to
// 1, 4: 736-775; 2, 4: 738; 4, 2: 775; 4, 4: 718; 8, 2: 851; the packed
// shared-memory pipeline: 870.
constexpr int kChainU = 2, kChainKB = 3;
// The same kernel without a chain is the vector combine of the flat and relay
// routes (more than 8 partners, or MOE_MOVE_VECTOR).  Four runs a lane and four
// partners a round took the flat combine 316.5 us at prefill-fp8 (the bulk
// pipeline 313.5) and 82.1 us at decode (84.9); cold, with L2 flushed before
// the call, the two match at decode, so the bulk pipeline stays the default.
constexpr int kFlatVecU = 4, kFlatVecKB = 4;

template <int ACC, int U, int KB, class Route>
__global__ void __launch_bounds__(kMoveThreads)
combine_chain_vec_kernel(const Route rt, const int nvec, const int nspan, const uint4* __restrict__ y,
                         uint4* __restrict__ out, float* __restrict__ acc_rows, bool acc_v8) {
    // Launched under programmatic dependent launch: nothing the previous
    // kernel writes (rows, the chain, positions) is read before this wait; a
    // CTA that has started lets the next kernel be scheduled.
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long units = rt.units() * nspan;
    const long long nw = (long long)gridDim.x * kMoveWarps;
    const uint64_t ypol = l2_evict_first_policy();  // y rows are read once
    for (long long u = (long long)blockIdx.x * kMoveWarps + (threadIdx.x >> 5); u < units; u += nw) {
        const long long ui = u / nspan;
        const int c = (int)(u - ui * nspan);
        int p, cp, n;
        float w, cw;
        rt.partner(ui, true, lane, p, w);
        compact_partners(lane, p, w, cp, cw, n);
        if (ACC == kAccMid && n == 0) continue;  // nothing to add: the chain stays
        const int v0 = c * 32 * U + lane;  // this lane's first 16-byte run of the row
        const size_t row = (size_t)rt.self_row(ui);
        float* arow = acc_rows + row * (size_t)nvec * 8;
        float acc[U][8];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int vi = v0 + 32 * i;
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[i][q] = 0.0f;
            if ((ACC == kAccMid || ACC == kAccLast) && vi < nvec) {
                if (acc_v8) {
                    ld_stream_v8f(arow + 8 * vi, acc[i]);
                } else {
                    const uint4 a0 = ld_stream_v4(reinterpret_cast<const uint4*>(arow + 8 * vi));
                    const uint4 a1 = ld_stream_v4(reinterpret_cast<const uint4*>(arow + 8 * vi + 4));
                    acc[i][0] = __uint_as_float(a0.x); acc[i][1] = __uint_as_float(a0.y);
                    acc[i][2] = __uint_as_float(a0.z); acc[i][3] = __uint_as_float(a0.w);
                    acc[i][4] = __uint_as_float(a1.x); acc[i][5] = __uint_as_float(a1.y);
                    acc[i][6] = __uint_as_float(a1.z); acc[i][7] = __uint_as_float(a1.w);
                }
            }
        }
        for (int jb = 0; jb < n; jb += KB) {
            uint4 v[KB][U];
            float wj[KB];
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                const int pj = __shfl_sync(kAll, cp, (jb + j) & 31);
                wj[j] = __shfl_sync(kAll, cw, (jb + j) & 31);
                const bool use = jb + j < n;
                const uint4* src = y + (size_t)(use ? pj : 0) * nvec;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    v[j][i] = make_uint4(0u, 0u, 0u, 0u);
                    if (use && v0 + 32 * i < nvec) v[j][i] = ld_stream_v4_hint(src + v0 + 32 * i, ypol);
                }
            }
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                if (jb + j >= n) break;
#pragma unroll
                for (int i = 0; i < U; ++i) fma_bf16x8(acc[i], wj[j], v[j][i]);
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int vi = v0 + 32 * i;
            if (vi >= nvec) continue;
            if constexpr (ACC == kAccFirst || ACC == kAccMid) {
                if (acc_v8) {
                    st_v8f(arow + 8 * vi, acc[i]);
                } else {
                    uint4* a4 = reinterpret_cast<uint4*>(arow + 8 * vi);
                    st_v4(a4, make_uint4(__float_as_uint(acc[i][0]), __float_as_uint(acc[i][1]),
                                         __float_as_uint(acc[i][2]), __float_as_uint(acc[i][3])));
                    st_v4(a4 + 1, make_uint4(__float_as_uint(acc[i][4]), __float_as_uint(acc[i][5]),
                                             __float_as_uint(acc[i][6]), __float_as_uint(acc[i][7])));
                }
            } else {
                st_v4(out + row * (size_t)nvec + vi, pack_bf16x8(acc[i]));
            }
        }
    }
}

// 32- or 16-byte pieces of a row, moved through registers.
template <int VB> struct VecT;
template <> struct VecT<32> {
    uint32_t w[8];
    __device__ __forceinline__ void load(const uint8_t* p) {
        asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                       "=r"(w[7])
                     : "l"(p));
    }
    __device__ __forceinline__ void store(uint8_t* p) const {
        asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                        "r"(w[7])
                     : "memory");
    }
};
template <> struct VecT<16> {
    uint32_t w[4];
    __device__ __forceinline__ void load(const uint8_t* p) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p));
    }
    __device__ __forceinline__ void store(uint8_t* p) const {
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                     :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
    }
};

// ---- quantise-in-dispatch ----------------------------------------------------

// bf16 rows in, e4m3 rows + fp32 scales out, one scale per 128 columns: the
// dispatch kernel converts to FP8 on its way ("Balancing and Beyond", section
// 3.1).  A warp takes one (token, span of 2048 columns) unit, two chunks of
// 1024 columns, and loads the whole span before it converts any of it: in
// chunk c, lane L holds columns 1024c + 32L .. 1024c + 32L + 31, so the four
// lanes 4g .. 4g+3 share scale group g of the chunk.  Per group: scale =
// amax / 448 (1 for an all-zero group), code = e4m3(x / scale) with
// round-to-nearest-even and saturation.  A lane's 32 codes go to every
// receive row of the token as one 32-byte store (two 16-byte ones when the
// rows are only 16-byte aligned), and the span's 16 scales as one request,
// lane g holding group g's.
constexpr int kQuantSpanCols = 2048;
constexpr int kQuantChunkCols = 1024;

template <int VB>
__global__ void __launch_bounds__(kMoveThreads)
dispatch_quant_kernel(const MoveArgs m, const uint8_t* __restrict__ x, uint8_t* __restrict__ recv,
                      float* __restrict__ rs, int h) {
    // Launched under programmatic dependent launch: the positions are read
    // after this wait; a CTA that has started lets the combine be scheduled.
    pdl_wait();
    pdl_launch_dependents();
    constexpr int NIN = 64 / VB;   // pieces of a lane's 32 bf16 inputs
    constexpr int NOUT = 32 / VB;  // pieces of its 32 codes
    constexpr unsigned kAll = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kMoveWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kMoveWarps;
    const int S = m.T * m.k;
    const int groups = h / 128;
    const long long units = (long long)m.T * m.nchunks;  // nchunks: spans per row here
    for (long long u = gwarp; u < units; u += nwarps) {
        const int t = (int)(u / m.nchunks);
        const int span = (int)(u - (long long)t * m.nchunks);
        int p = -1;
        if (lane < m.k) {
            p = m.pos[(size_t)t * m.k + lane];
            if (p < 0 || p >= S) p = -1;
        }
        VecT<VB> v[2][NIN];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int col = span * kQuantSpanCols + c * kQuantChunkCols + lane * 32;
            if (col < h) {  // h % 128 == 0: groups are whole
                const uint8_t* src = x + ((size_t)t * h + col) * 2;
#pragma unroll
                for (int i = 0; i < NIN; ++i) v[c][i].load(src + i * VB);
            } else {
#pragma unroll
                for (int i = 0; i < NIN; ++i)
#pragma unroll
                    for (int w = 0; w < VB / 4; ++w) v[c][i].w[w] = 0u;
            }
        }
        float my_scale = 1.0f;  // lanes 0..15: the scale of the span's group `lane`
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int col = span * kQuantSpanCols + c * kQuantChunkCols + lane * 32;
            const bool active = col < h;
            if (!__any_sync(kAll, active)) break;  // past the row's end for the whole warp
            float f[32];
#pragma unroll
            for (int i = 0; i < NIN; ++i)
#pragma unroll
                for (int w = 0; w < VB / 4; ++w) {
                    const uint32_t q = v[c][i].w[w];
                    f[2 * (i * (VB / 4) + w)] = __uint_as_float(q << 16);
                    f[2 * (i * (VB / 4) + w) + 1] = __uint_as_float(q & 0xffff0000u);
                }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 2));
            const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            // lane c*8 + g keeps the scale of the chunk's group g (held by lanes 4g .. 4g+3)
            const float sg = __shfl_sync(kAll, scale, 4 * (lane & 7));
            if ((lane >> 3) == c) my_scale = sg;
            VecT<VB> codes[NOUT];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(f[4 * i] / scale, f[4 * i + 1] / scale), __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(f[4 * i + 2] / scale, f[4 * i + 3] / scale), __NV_SATFINITE, __NV_E4M3);
                codes[i / (VB / 4)].w[i % (VB / 4)] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            for (int j = 0; j < m.k; ++j) {
                const int pj = __shfl_sync(kAll, p, j);
                if (pj < 0 || !active) continue;
                uint8_t* dst = recv + (size_t)pj * h + col;
#pragma unroll
                for (int i = 0; i < NOUT; ++i) codes[i].store(dst + i * VB);
            }
        }
        const int g = span * (kQuantSpanCols / 128) + lane;  // the span's group `lane`
        const bool has_group = lane < kQuantSpanCols / 128 && g < groups;
        for (int j = 0; j < m.k; ++j) {
            const int pj = __shfl_sync(kAll, p, j);
            if (pj >= 0 && has_group) rs[(size_t)pj * groups + g] = my_scale;
        }
    }
}

// ---- bulk (TMA) kernels --------------------------------------------------

// Device fault bits of the row movers (bounded waits that gave up).
__device__ unsigned int g_move_faults;
constexpr unsigned kFaultWaitTimeout = 0x1u;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

// Per-warp pipeline bookkeeping: a stage is "pending" from the copy issue
// until its barrier phase is waited for; ph counts completed waits, so the
// phase to wait for has parity ph & 1.
template <int STAGES>
__device__ __forceinline__ void drain_stages(uint32_t bar0, const bool (&pending)[STAGES],
                                             const uint32_t (&ph)[STAGES]) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s)
        if (pending[s]) mbar_wait_bounded(bar0 + 8 * s, ph[s] & 1u, kWaitLimitNs);
}

// Combine: each warp owns STAGES stages of KMAX rows x CHUNK bytes; a stage
// holds the partner row pieces (at most KMAX) of one (unit, column chunk).
// Plain: the partners are summed into the unit's own row.  GROUPED: partners
// with the same key are summed into output row `key` (one sum per key, each
// in ascending lane order).
template <int WARPS, int STAGES, int CHUNK, int KMAX, bool GROUPED, class Route>
__global__ void __launch_bounds__(WARPS * 32, 1)
combine_bulk_kernel(const Route rt, const int nch, const uint8_t* __restrict__ y,
                    uint8_t* __restrict__ out, int row_bytes) {
    constexpr int STAGE_BYTES = KMAX * CHUNK;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar[WARPS][STAGES];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t stage0 = smem_u32(smem + (size_t)warp * STAGES * STAGE_BYTES);
    const uint32_t bar0 = smem_u32(&s_bar[warp][0]);
    const uint64_t ypol = l2_evict_first_policy();  // y rows are read once
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    // Launched under programmatic dependent launch: the CTAs may become
    // resident while the previous kernel drains; nothing it writes (rows,
    // positions) is read before this wait.
    pdl_wait();
    __syncwarp();

    const long long units = rt.units() * nch;
    const long long nw = (long long)gridDim.x * WARPS;
    const long long gw = (long long)blockIdx.x * WARPS + warp;

    long long su[STAGES];   // (unit, chunk) held by each stage
    unsigned vm[STAGES];    // partner rows of that unit that were fetched
    float wr[STAGES];       // lane j: weight of partner j of that unit
    int kr[STAGES];         // GROUPED, lane j: output row of partner j
    unsigned gr[STAGES];    // GROUPED, lane j: partners sharing that output row
    bool pending[STAGES];
    uint32_t ph[STAGES];

    auto fetch_meta = [&](long long u, int& p, float& wv, int& kk) {
        rt.partner(u / nch, u < units, lane, p, wv);
        kk = -1;
        if constexpr (GROUPED) {
            kk = rt.key(u / nch, u < units, lane);
            if (kk < 0) p = -1;
        }
        if (lane >= KMAX) p = -1;  // routes launched here have at most KMAX partners
    };
    // Issues the partner bulk copies of unit u into stage s (all lanes call it).
    auto issue = [&](int s, long long u, int p) -> unsigned {
        const int c = (int)(u % nch);
        const int cb = min(CHUNK, row_bytes - c * CHUNK);
        const unsigned mask = __ballot_sync(0xffffffffu, p >= 0);
        if (lane == 0) mbar_arrive_expect_tx(bar0 + 8 * s, (uint32_t)(__popc(mask) * cb));
        __syncwarp();
        if (p >= 0) {
            const uint8_t* src = y + (size_t)p * row_bytes + (size_t)c * CHUNK;
            // The grouped pass (relay hop 1) loads plainly: the partial rows it
            // writes are read back by the next pass, and they stay in L2 more
            // often that way (1 % faster relay step on GB300).
            if constexpr (GROUPED)
                bulk_g2s(stage0 + s * STAGE_BYTES + lane * CHUNK, src, (uint32_t)cb, bar0 + 8 * s);
            else
                bulk_g2s_hint(stage0 + s * STAGE_BYTES + lane * CHUNK, src, (uint32_t)cb, bar0 + 8 * s, ypol);
        }
        return mask;
    };

#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        su[s] = gw + s * nw;
        ph[s] = 0;
        pending[s] = su[s] < units;
        int p, kk;
        float wv;
        fetch_meta(su[s], p, wv, kk);
        wr[s] = wv;
        kr[s] = kk;
        gr[s] = GROUPED ? __match_any_sync(0xffffffffu, p >= 0 ? kk : -1) : 0u;
        vm[s] = pending[s] ? issue(s, su[s], p) : 0u;
    }
    bool failed = false, busy = true;
    while (busy && !failed) {
        busy = false;
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            if (!pending[s] || failed) continue;
            const long long u = su[s];
            const long long un = u + STAGES * nw;
            int pn, kn;
            float wn;
            fetch_meta(un, pn, wn, kn);  // overlaps the wait below
            // give up as a warp, so that no lane runs ahead into a shuffle
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * s, ph[s] & 1u, kWaitLimitNs))) {
                failed = true;
                continue;
            }
            ph[s] += 1;
            pending[s] = false;
            const long long ui = u / nch;
            const int c = (int)(u - ui * nch);
            const int cb = min(CHUNK, row_bytes - c * CHUNK);
            float wj[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) wj[j] = __shfl_sync(0xffffffffu, wr[s], j);
            const uint32_t st = stage0 + s * STAGE_BYTES;
            // one output row per group of partners (a single group when not GROUPED)
            unsigned rem = vm[s];
            bool first = true;
            while (GROUPED ? rem != 0u : first) {
                first = false;
                unsigned grp = rem;
                int orow_i = rt.self_row(ui);
                if constexpr (GROUPED) {
                    const int lead = __ffs(rem) - 1;
                    grp = __shfl_sync(0xffffffffu, gr[s], lead) & rem;
                    orow_i = __shfl_sync(0xffffffffu, kr[s], lead);
                }
                rem &= ~grp;
                uint4* orow = reinterpret_cast<uint4*>(out + (size_t)orow_i * row_bytes + (size_t)c * CHUNK);
                for (int v = lane; v < cb / 16; v += 32) {
                    float acc[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if ((grp >> j) & 1u) fma_bf16x8(acc, wj[j], lds_v4(st + j * CHUNK + v * 16));
                    st_v4(orow + v, pack_bf16x8(acc));
                }
            }
            __syncwarp();
            fence_proxy_async_smem();
            su[s] = un;
            wr[s] = wn;
            kr[s] = kn;
            gr[s] = GROUPED ? __match_any_sync(0xffffffffu, pn >= 0 ? kn : -1) : 0u;
            if (un < units) {
                vm[s] = issue(s, un, pn);
                pending[s] = true;
                busy = true;
            }
        }
    }
    if (failed) {
        if (lane == 0) atomicOr(&g_move_faults, kFaultWaitTimeout);
        drain_stages<STAGES>(bar0, pending, ph);
    }
}

// Packed combine: a stage holds kPackSlots pieces of kPiece bytes, filled
// with as many column pieces of the unit's partners as fit.  A unit is
// (output row, span of kPackSlots pieces); with n partners a round takes
// `per` pieces of every partner (per = floor(kPackSlots / n)), so a unit with
// one or two partners fills its stages as fully as one with eight.  Rounds
// flow in order through the warp's stages; the partners of the next unit are
// looked up while the current unit's rounds are in flight.
//
// ACC carries an fp32 chain across launches (kAcc*): the first group writes
// it, middle groups read and write it, the last reads it and writes the bf16
// row.  Chain values are read from registers' view of 32 contiguous bytes a
// lane and written as 32-byte stores (16-byte halves when the chain is only
// 16-byte aligned).  Bringing them through the stage (a separate chain area
// after the y slots, so half the stages fit an SM) and prefetching a whole
// round into registers (two CTAs of 8 warps instead of three) both measured
// slower.  At most kPackSlots partners (compacted, ascending lane order, so
// each sum keeps the route's partner order).
constexpr int kPiece = 512, kPackSlots = 8;
constexpr int kCombCtasPerSmPacked = 3;  // first group: registers capped so that 3 CTAs of 8 warps fit an SM

template <int ACC> struct PackedShape {
    static constexpr bool kChainIn = ACC == kAccMid || ACC == kAccLast;
    static constexpr int kWarps = 8, kStages = 2, kCtasPerSm = kCombCtasPerSmPacked;
    static constexpr int kStageBytes = kPackSlots * kPiece;
};


template <int ACC, class Route>
__global__ void __launch_bounds__(PackedShape<ACC>::kWarps * 32, PackedShape<ACC>::kCtasPerSm)
combine_packed_kernel(const Route rt, const uint8_t* __restrict__ y, uint8_t* __restrict__ out, int row_bytes,
                      float* __restrict__ acc_rows, bool acc_v8) {
    using Sh = PackedShape<ACC>;
    constexpr int WARPS = Sh::kWarps, STAGES = Sh::kStages, STAGE_BYTES = Sh::kStageBytes;
    constexpr bool CHAIN_IN = Sh::kChainIn;
    constexpr bool CHAIN_AHEAD = ACC == kAccMid;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar[WARPS][STAGES];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t stage0 = smem_u32(smem + (size_t)warp * STAGES * STAGE_BYTES);
    const uint32_t bar0 = smem_u32(&s_bar[warp][0]);
    const uint64_t ypol = l2_evict_first_policy();  // y rows are read once
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int npieces = (row_bytes + kPiece - 1) / kPiece;      // pieces per row
    const int nspan = (npieces + kPackSlots - 1) / kPackSlots;  // spans per row
    const long long units = rt.units() * nspan;
    const long long nw = (long long)gridDim.x * WARPS;
    const long long gw = (long long)blockIdx.x * WARPS + warp;
    const size_t chain_row = (size_t)(row_bytes / 2);           // floats of a chain row

    // The unit whose rounds are being issued, and the next one.
    struct Meta {
        long long u;
        int p;     // lane j < n: row of partner j
        float w;   // lane j < n: its weight
        int n;     // partners
        int per;   // pieces of each partner per round
        int rounds;
    };
    auto fetch = [&](long long u) {
        Meta m;
        m.u = u;
        int p;
        float w;
        rt.partner(u / nspan, u < units, lane, p, w);
        if (lane >= kPackSlots) p = -1;
        compact_partners(lane, p, w, m.p, m.w, m.n);
        const int span = (int)(u % nspan);
        const int cnt = min(kPackSlots, npieces - span * kPackSlots);  // pieces in this span
        m.per = m.n > 0 ? kPackSlots / m.n : kPackSlots;
        const bool skip = ACC == kAccMid && m.n == 0;  // nothing to add: the chain stays
        m.rounds = (u < units && !skip) ? (cnt + m.per - 1) / m.per : 0;
        return m;
    };

    // per stage: unit, first piece, pieces, partners, weights
    long long su[STAGES];
    int sp0[STAGES], scnt[STAGES], sn[STAGES];
    float sw[STAGES];
    bool pending[STAGES];
    uint32_t ph[STAGES];

    Meta cur = fetch(gw), nxt = fetch(gw + nw);
    int cround = 0;
    // Skips units with no rounds; false when the warp has no item left.
    auto settle = [&]() -> bool {
        while (cur.u < units && cround >= cur.rounds) {
            cur = nxt;
            nxt = fetch(cur.u + nw);
            cround = 0;
        }
        return cur.u < units;
    };
    // Issues the next round of the current unit into stage s (all lanes).
    auto issue = [&](int s) {
        const int span = (int)(cur.u % nspan);
        const int first = span * kPackSlots + cround * cur.per;  // first piece of the round
        const int cnt = min(cur.per, min(kPackSlots, npieces - span * kPackSlots) - cround * cur.per);
        su[s] = cur.u;
        sp0[s] = first;
        scnt[s] = cnt;
        sn[s] = cur.n;
        sw[s] = cur.w;
        // lane L < cnt * n copies piece first + L / n of partner L % n into slot L
        const int j = cur.n > 0 ? lane % cur.n : 0;
        const int pj = __shfl_sync(kAll, cur.p, j);
        uint32_t bytes = 0;
        for (int i = 0; i < cnt; ++i) bytes += (uint32_t)min(kPiece, row_bytes - (first + i) * kPiece);
        if (lane == 0) mbar_arrive_expect_tx(bar0 + 8 * s, bytes * (uint32_t)cur.n);
        __syncwarp();
        if (lane < cnt * cur.n) {
            const int piece = first + lane / cur.n;
            const int pb = min(kPiece, row_bytes - piece * kPiece);
            bulk_g2s_hint(stage0 + s * STAGE_BYTES + lane * kPiece,
                          y + (size_t)pj * row_bytes + (size_t)piece * kPiece, (uint32_t)pb, bar0 + 8 * s, ypol);
        }
        cround += 1;
    };

#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        ph[s] = 0;
        pending[s] = settle();
        if (pending[s]) issue(s);
    }
    bool failed = false, busy = true;
    while (busy && !failed) {
        busy = false;
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            if (!pending[s] || failed) continue;
            const int n = sn[s];
            const long long orow = rt.self_row(su[s] / nspan);
            // Middle groups load the chain values of the round's first piece
            // before the wait for the stage, and those of piece i + 1 before
            // piece i is summed and stored, so each load's latency overlaps other
            // work (G = 4 at prefill-fp8 on GB300: the two middle groups 208.9 and
            // 213.0 -> 196.6 and 204.8 us).  The last group, with about twice the
            // partners, loads each piece's values straight into its sums inside
            // the lane guard (ahead, or loaded outside the guard, it took 319.5
            // instead of 303-305 us).  The piece loop is left to the compiler:
            // unrolled over pieces and partners the code outgrows the instruction
            // cache (a first group ran 1.6 times slower).
            const float* chain0 = acc_rows + (size_t)orow * chain_row + 8 * lane;
            auto load_chain = [&](int piece, float (&c)[8]) {
                if (lane < min(kPiece, row_bytes - piece * kPiece) / 16) {
                    const float* a = chain0 + (size_t)piece * (kPiece / 2);
                    if (acc_v8) {
                        ld_stream_v8f(a, c);
                    } else {
                        const uint4 a0 = ld_stream_v4(reinterpret_cast<const uint4*>(a));
                        const uint4 a1 = ld_stream_v4(reinterpret_cast<const uint4*>(a + 4));
                        c[0] = __uint_as_float(a0.x); c[1] = __uint_as_float(a0.y);
                        c[2] = __uint_as_float(a0.z); c[3] = __uint_as_float(a0.w);
                        c[4] = __uint_as_float(a1.x); c[5] = __uint_as_float(a1.y);
                        c[6] = __uint_as_float(a1.z); c[7] = __uint_as_float(a1.w);
                    }
                }
            };
            float chain_next[8];
            if constexpr (CHAIN_AHEAD) load_chain(sp0[s], chain_next);
            if (!__all_sync(kAll, mbar_wait_bounded(bar0 + 8 * s, ph[s] & 1u, kWaitLimitNs))) {
                failed = true;
                continue;
            }
            ph[s] += 1;
            pending[s] = false;
            const uint32_t st = stage0 + s * STAGE_BYTES;
            float wj[kPackSlots];
#pragma unroll
            for (int j = 0; j < kPackSlots; ++j) wj[j] = __shfl_sync(kAll, sw[s], j);
            for (int i = 0; i < scnt[s]; ++i) {
                const int piece = sp0[s] + i;
                const int pb = min(kPiece, row_bytes - piece * kPiece);
                uint4* o = reinterpret_cast<uint4*>(out + (size_t)orow * row_bytes + (size_t)piece * kPiece);
                float* arow = ACC == kAccNone ? nullptr : acc_rows + (size_t)orow * chain_row + (size_t)piece * (kPiece / 2);
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = CHAIN_AHEAD ? chain_next[q] : 0.0f;
                if (CHAIN_AHEAD && i + 1 < scnt[s]) load_chain(piece + 1, chain_next);
                // Lane v's 8 chain values are 32 contiguous bytes.
                if (lane < pb / 16) {
                    const int v = lane;
                    if (CHAIN_IN && !CHAIN_AHEAD) {
                        if (acc_v8) {
                            ld_stream_v8f(arow + 8 * v, acc);
                        } else {
                            const uint4 a0 = ld_stream_v4(reinterpret_cast<const uint4*>(arow + 8 * v));
                            const uint4 a1 = ld_stream_v4(reinterpret_cast<const uint4*>(arow + 8 * v + 4));
                            acc[0] = __uint_as_float(a0.x); acc[1] = __uint_as_float(a0.y);
                            acc[2] = __uint_as_float(a0.z); acc[3] = __uint_as_float(a0.w);
                            acc[4] = __uint_as_float(a1.x); acc[5] = __uint_as_float(a1.y);
                            acc[6] = __uint_as_float(a1.z); acc[7] = __uint_as_float(a1.w);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kPackSlots; ++j)
                        if (j < n) fma_bf16x8(acc, wj[j], lds_v4(st + (i * n + j) * kPiece + v * 16));
                    if constexpr (ACC == kAccFirst || ACC == kAccMid) {
                        // with a 32-byte aligned chain, one 256-bit store: a warp
                        // request covers 1 KB of whole sectors
                        if (acc_v8) {
                            st_v8f(arow + 8 * v, acc);
                        } else {
                            uint4* a4 = reinterpret_cast<uint4*>(arow + 8 * v);
                            st_v4(a4, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                                 __float_as_uint(acc[2]), __float_as_uint(acc[3])));
                            st_v4(a4 + 1, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                                     __float_as_uint(acc[6]), __float_as_uint(acc[7])));
                        }
                    } else {
                        st_v4(o + v, pack_bf16x8(acc));
                    }
                }
            }
            __syncwarp();
            fence_proxy_async_smem();
            if (settle()) {
                issue(s);
                pending[s] = true;
                busy = true;
            }
        }
    }
    if (failed) {
        if (lane == 0) atomicOr(&g_move_faults, kFaultWaitTimeout);
        drain_stages<STAGES>(bar0, pending, ph);
    }
}

// Dispatch through shared memory: each warp owns `stages` stages of `chunk`
// bytes of source rows (warps, stages and chunk are launch values); a stage
// holds one (unit, column chunk), written to the unit's partner rows by one
// bulk store each.  fp8 scale rows (`groups` floats) travel with the first
// chunk: through the stage as one more bulk load and a bulk store per partner
// when sbytes = 4 * groups > 0 (a multiple of 16 bytes, both arrays 16-byte
// aligned), otherwise by plain 4-byte copies.  SKIP_EMPTY (routes where many
// units have no partner, such as one expert group): partners are looked up
// before the load, and a unit without any is not loaded.  Dynamic shared
// memory: the barriers (kDispBarBytes), then the warps' stages.
constexpr int kMaxDispWarps = 16, kMaxDispStages = 8;
constexpr int kDispBarBytes = kMaxDispWarps * kMaxDispStages * 8;

template <class Route, bool SKIP_EMPTY = false>
__global__ void __launch_bounds__(kMaxDispWarps * 32, 1)
dispatch_bulk_kernel(const Route rt, const int nch, const int stages, const int chunk, const uint8_t* __restrict__ x,
                     const float* __restrict__ xs, uint8_t* __restrict__ recv, float* __restrict__ rs, int row_bytes,
                     int groups, int sbytes) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
    const int stride = chunk + sbytes;  // a stage: the chunk, then the scale row
    const uint32_t stage0 = smem_u32(smem + kDispBarBytes + (size_t)warp * stages * stride);
    const uint32_t bar0 = smem_u32(smem + 8 * kMaxDispStages * warp);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const long long units = rt.units() * nch;
    const long long nw = (long long)gridDim.x * warps;
    const long long gw = (long long)blockIdx.x * warps + warp;
    const long long step = (long long)stages * nw;  // a stage's stride through the units

    long long su[kMaxDispStages];
    bool pending[kMaxDispStages];
    uint32_t ph[kMaxDispStages];
    int pr[kMaxDispStages];  // SKIP_EMPTY: this lane's partner row of the stage's unit
    // Issues the bulk load of unit u into stage s (lane 0); with SKIP_EMPTY
    // (all lanes call it) returns false, loading nothing, when u has no partner.
    auto issue = [&](int s, long long u, int& p_out) -> bool {
        const long long ui = u / nch;
        if constexpr (SKIP_EMPTY) {
            float unused;
            rt.partner(ui, true, lane, p_out, unused);
            if (__ballot_sync(0xffffffffu, p_out >= 0) == 0u) return false;
        }
        if (lane == 0) {
            const int c = (int)(u - ui * nch);
            const int cb = min(chunk, row_bytes - c * chunk);
            const bool with_scales = sbytes > 0 && c == 0;
            const size_t src = (size_t)rt.self_row(ui);
            mbar_arrive_expect_tx(bar0 + 8 * s, (uint32_t)(cb + (with_scales ? sbytes : 0)));
            bulk_g2s(stage0 + s * stride, x + src * row_bytes + (size_t)c * chunk, (uint32_t)cb, bar0 + 8 * s);
            if (with_scales)
                bulk_g2s(stage0 + s * stride + chunk, xs + src * groups, (uint32_t)sbytes, bar0 + 8 * s);
        }
        return true;
    };
    // First unit at or after u, in this stage's stride, that needs a load.
    auto next_loaded = [&](int s, long long u, int& p_out) -> long long {
        while (u < units && !issue(s, u, p_out)) u += step;
        return u;
    };

#pragma unroll
    for (int s = 0; s < kMaxDispStages; ++s) {
        pending[s] = false;
        ph[s] = 0;
        pr[s] = -1;
        su[s] = units;
        if (s < stages) {
            su[s] = next_loaded(s, gw + s * nw, pr[s]);
            pending[s] = su[s] < units;
        }
    }
    bool failed = false, busy = true;
    while (busy && !failed) {
        busy = false;
#pragma unroll
        for (int s = 0; s < kMaxDispStages; ++s) {
            if (!pending[s] || failed) continue;
            const long long u = su[s];
            const long long ui = u / nch;
            const int c = (int)(u - ui * nch);
            const int cb = min(chunk, row_bytes - c * chunk);
            int p = pr[s];
            if constexpr (!SKIP_EMPTY) {
                float unused;
                rt.partner(ui, true, lane, p, unused);
            }
            // give up as a warp, so that no lane runs ahead into a shuffle
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * s, ph[s] & 1u, kWaitLimitNs))) {
                failed = true;
                continue;
            }
            ph[s] += 1;
            pending[s] = false;
            fence_proxy_async_smem();
            if (p >= 0) {
                bulk_s2g(recv + (size_t)p * row_bytes + (size_t)c * chunk, stage0 + s * stride, (uint32_t)cb);
                if (sbytes > 0 && c == 0)
                    bulk_s2g(rs + (size_t)p * groups, stage0 + s * stride + chunk, (uint32_t)sbytes);
            }
            bulk_commit();
            if (groups > 0 && sbytes == 0 && c == 0) {
                // fp8 scales that a bulk copy cannot move: plain copies with the first chunk.
                const size_t src = (size_t)rt.self_row(ui) * groups;
                for (unsigned mm = __ballot_sync(0xffffffffu, p >= 0); mm; mm &= mm - 1) {
                    const int pj = __shfl_sync(0xffffffffu, p, __ffs(mm) - 1);
                    for (int g = lane; g < groups; g += 32) rs[(size_t)pj * groups + g] = xs[src + g];
                }
            }
            // The stage may be refilled once every lane's stores have read it.
            bulk_wait_read<0>();
            __syncwarp();
            su[s] = next_loaded(s, u + step, pr[s]);
            if (su[s] < units) {
                pending[s] = true;
                busy = true;
            }
        }
    }
    bulk_wait_all();
    if (failed) {
        if (lane == 0) atomicOr(&g_move_faults, kFaultWaitTimeout);
#pragma unroll
        for (int s = 0; s < kMaxDispStages; ++s)
            if (pending[s]) mbar_wait_bounded(bar0 + 8 * s, ph[s] & 1u, kWaitLimitNs);
    }
}

// ---- vector dispatch ---------------------------------------------------------
//
// Rows through registers: one warp per (unit, span of the source row).  Every
// lane loads its V vectors of VB bytes of the span, all loads issued before
// any store, then writes them to each partner row in ascending lane order.  A
// span is 32 x V x VB = 7168 bytes (an fp8 row of h = 7168; half a bf16 one).
// With VB = 32 the loads and stores are 256-bit (sm_100 and later), so a warp
// request covers 1 KB of whole sectors.  On GB300 this moved a read-1 /
// write-8 broadcast of 16384 fp8 rows (7168 B, random receive rows) in
// 166-168 us against 182-184 us for the shared-memory bulk pipeline, and
// 4096 bf16 rows in 86-88 us against 94 us: with the same bytes in flight per
// SM, the register path keeps the DRAM write stream fuller.  fp8 scale rows travel
// with the first span: as 32-byte pieces, one a lane, when the row is whole
// pieces and both scale arrays are 32-byte aligned; otherwise lane L keeps
// words L + 32 q (rows of up to 32 x kVecScaleWords groups; longer ones are
// copied word by word).  A unit without partners loads nothing.
constexpr int kVecThreads = 256;
constexpr int kVecMinBlocks = 2;   // ~100 registers a thread: two 8-warp CTAs fill an SM's registers
constexpr int kVecScaleWords = 4;
// A grid of 8x the resident CTAs, each warp taking one or two units, moved
// the fp8 broadcast above in 166-168 us on GB300; a persistent grid of
// exactly the resident CTAs looping over the units took 185 us.
constexpr int kVecOversubscribe = 8;

template <int VB> struct VecSpan { static constexpr int V = 7168 / (32 * VB); };

template <int VB, class Route>
__global__ void __launch_bounds__(kVecThreads, kVecMinBlocks)
dispatch_vec_kernel(const Route rt, const int nspan, const uint8_t* __restrict__ x, const float* __restrict__ xs,
                    uint8_t* __restrict__ recv, float* __restrict__ rs, int row_bytes, int groups, bool scale_v8) {
    // Launched under programmatic dependent launch: the CTAs may become
    // resident while the previous kernel (the layout) finishes; every read of
    // its positions comes after this wait.  A CTA that has started lets the
    // next kernel (the combine) be scheduled: its CTAs take the room of
    // finished ones in the last wave and wait for this grid's end.
    pdl_wait();
    pdl_launch_dependents();
    constexpr int V = VecSpan<VB>::V;
    constexpr int SPAN = 32 * V * VB;
    constexpr int WPB = kVecThreads / 32;
    const int lane = threadIdx.x & 31;
    const long long units = rt.units() * nspan;
    const long long nw = (long long)gridDim.x * WPB;
    long long u = (long long)blockIdx.x * WPB + (threadIdx.x >> 5);
    // partners of the warp's next unit, looked up one unit ahead: the loads
    // go out a unit early and are used only when that unit's turn comes
    RawPartner next = rt.raw(u / nspan, u < units, lane);
    for (; u < units; u += nw) {
        const long long ui = u / nspan;
        const int c = (int)(u - ui * nspan);
        int p;
        float unused;
        rt.resolve(next, p, unused);
        next = rt.raw((u + nw) / nspan, u + nw < units, lane);
        const unsigned pm = __ballot_sync(kAll, p >= 0);
        if (pm == 0u) continue;  // nothing to write
        const size_t srow = (size_t)rt.self_row(ui);
        const uint8_t* src = x + srow * row_bytes + (size_t)c * SPAN;
        const int lim = row_bytes - c * SPAN;  // bytes of the row from this span on
        VecT<VB> v[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int off = (i * 32 + lane) * VB;
            if (off < lim) v[i].load(src + off);
        }
        const bool scales = groups > 0 && c == 0;
        // a scale row of 32-byte pieces (groups % 8 == 0, both arrays 32-byte
        // aligned, at most 32 pieces) moves as one 256-bit vector a lane
        const bool keep = groups <= 32 * kVecScaleWords;
        const int svec = scale_v8 ? groups / 8 : 0;
        float sv[kVecScaleWords];
        VecT<32> s8;
        if (scales && scale_v8 && lane < svec) s8.load(reinterpret_cast<const uint8_t*>(xs + srow * groups) + 32 * lane);
#pragma unroll
        for (int q = 0; q < kVecScaleWords; ++q)
            sv[q] = (scales && !scale_v8 && keep && lane + 32 * q < groups) ? xs[srow * groups + lane + 32 * q] : 0.0f;
        for (unsigned m = pm; m; m &= m - 1) {
            const int pj = __shfl_sync(kAll, p, __ffs(m) - 1);
            uint8_t* dst = recv + (size_t)pj * row_bytes + (size_t)c * SPAN;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int off = (i * 32 + lane) * VB;
                if (off < lim) v[i].store(dst + off);
            }
            if (scales) {
                float* srow_out = rs + (size_t)pj * groups;
                if (scale_v8) {
                    if (lane < svec) s8.store(reinterpret_cast<uint8_t*>(srow_out) + 32 * lane);
                } else if (keep) {
#pragma unroll
                    for (int q = 0; q < kVecScaleWords; ++q)
                        if (lane + 32 * q < groups) srow_out[lane + 32 * q] = sv[q];
                } else {
                    for (int g = lane; g < groups; g += 32) srow_out[g] = xs[srow * groups + g];
                }
            }
        }
    }
}

template <typename K>
int resident_blocks(K kernel) {
    return device_sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kernel), kMoveThreads, 0);
}

template <typename K>
int grid_for(K kernel, long long units) {
    const long long need = (units + kMoveWarps - 1) / kMoveWarps;
    const long long cap = resident_blocks(kernel);
    return (int)max(1LL, min(need, cap));
}

// SMs a mover's grid may cover: the tuning's count, at most the GPU's.
int mover_sms(int want) {
    const int sms = device_sm_count();
    return want > 0 && want < sms ? want : sms;
}

// Grid of `per_sm` CTAs on each of `sms` SMs, no larger than the work needs.
int capped_grid(long long units, int warps_per_cta, int sms, int per_sm) {
    const long long need = (units + warps_per_cta - 1) / warps_per_cta;
    const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
    return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

// Default shapes of the bulk pipelines, chosen by a sweep on GB300 at the
// prefill-fp8 shape: warps per CTA, stages per warp, chunk bytes, CTAs per SM.
constexpr int kCombWarps = 8, kCombStages = 2, kCombChunk = 512, kCombCtasPerSm = 3;
constexpr int kDispWarps = 4, kDispStages = 4, kDispChunk = 7168;
// Dispatch routes whose units have few partners (the relay hops: 2-4 rows a
// unit at the decode and prefill shapes; one expert group: about k/G) issue
// fewer stores per load, so more warps keep more loads in flight: 6 warps of
// 4 stages made a graph-replayed relay step 7 % faster at decode (360.8 ->
// 334.5 us) and the G = 4 group schedule 2.6-3.5 % faster, while the flat
// dispatch (8 partners) was 0.4-0.7 % slower with them.
constexpr int kFewWarps = 6, kFewStages = 4;
// Shared memory a dispatch CTA's stages may take: scale rows go through the
// stages only while every stage, chunk and scale row, fits in it.
constexpr size_t kDispSmemMax = 220 * 1024;

template <int WARPS, int STAGES, int CHUNK, int KMAX, bool GROUPED, int PER_SM, class Route>
cudaError_t launch_combine_bulk(const Route& rt, long long max_units, int nvec, const void* y, void* out,
                                const MoveShape& sh, cudaStream_t stream) {
    const int row_bytes = nvec * 16;
    const int nch = (row_bytes + CHUNK - 1) / CHUNK;
    const long long units = max_units * nch;
    if (units == 0) return cudaSuccess;
    auto kern = combine_bulk_kernel<WARPS, STAGES, CHUNK, KMAX, GROUPED, Route>;
    const size_t smem = (size_t)WARPS * STAGES * KMAX * CHUNK;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int grid = capped_grid(units, WARPS, mover_sms(sh.combine_sms), sh.combine_ctas > 0 ? sh.combine_ctas : PER_SM);
    return launch_pdl(kern, dim3(grid), dim3(WARPS * 32), smem, stream, rt, nch, static_cast<const uint8_t*>(y),
                      static_cast<uint8_t*>(out), row_bytes);
}

// The dispatch pipelines for one route.  kind: MOE_MOVE_VECTOR or
// MOE_MOVE_BULK (the caller resolves MOE_MOVE_AUTO); few: the route's units
// have few partners (bulk default: 6 warps per CTA instead of 4).
template <class Route, bool SKIP_EMPTY>
cudaError_t launch_dispatch_route(const Route& rt, long long max_units, int row_bytes, const void* x, const float* xs,
                                  void* dst, float* ds, int groups, const MoveShape& sh, int kind, bool few,
                                  cudaStream_t stream) {
    if (max_units == 0) return cudaSuccess;
    const int sms = mover_sms(sh.dispatch_sms);
    if (kind == MOE_MOVE_VECTOR) {
        // 32-byte vectors when every row and both bases allow them
        const bool v32 = row_bytes % 32 == 0 && (reinterpret_cast<uintptr_t>(x) & 31) == 0 &&
                         (reinterpret_cast<uintptr_t>(dst) & 31) == 0;
        const int span = 7168;
        const int nspan = (row_bytes + span - 1) / span;
        const long long units = max_units * nspan;
        // By default the grid holds up to kVecOversubscribe times the CTAs that
        // fit at once (about one unit per warp at the workloads here); a tuning
        // that sets SMs or CTAs per SM gets a persistent grid of that size.
        const bool persistent = sh.dispatch_sms > 0 || sh.dispatch_ctas > 0;
        const bool scale_v8 = groups > 0 && groups % 8 == 0 && groups / 8 <= 32 &&
                              (reinterpret_cast<uintptr_t>(xs) & 31) == 0 && (reinterpret_cast<uintptr_t>(ds) & 31) == 0;
        auto launch = [&](auto kern) {
            const int occ = blocks_per_sm(reinterpret_cast<const void*>(kern), kVecThreads, 0);
            const int per_sm = persistent ? (sh.dispatch_ctas > 0 ? min(sh.dispatch_ctas, occ) : occ)
                                          : occ * kVecOversubscribe;
            // programmatic dependent launch: the CTAs may become resident while
            // the previous kernel in the stream (the layout) finishes
            return launch_pdl(kern, dim3(capped_grid(units, kVecThreads / 32, sms, per_sm)), dim3(kVecThreads), 0,
                              stream, rt, nspan, static_cast<const uint8_t*>(x), xs, static_cast<uint8_t*>(dst), ds,
                              row_bytes, groups, scale_v8);
        };
        return v32 ? launch(dispatch_vec_kernel<32, Route>) : launch(dispatch_vec_kernel<16, Route>);
    }
    const int warps = sh.dispatch_warps > 0 ? sh.dispatch_warps : (few ? kFewWarps : kDispWarps);
    const int stages = sh.dispatch_stages > 0 ? sh.dispatch_stages : (few ? kFewStages : kDispStages);
    const int chunk = sh.dispatch_chunk > 0 ? sh.dispatch_chunk : kDispChunk;
    const int nch = (row_bytes + chunk - 1) / chunk;
    const long long units = max_units * nch;
    auto kern = dispatch_bulk_kernel<Route, SKIP_EMPTY>;
    // scale rows through the stages when a bulk copy can move them and they fit
    const int sbytes = (groups > 0 && groups % 4 == 0 &&
                        (size_t)warps * stages * (chunk + 4 * (size_t)groups) <= kDispSmemMax &&
                        (reinterpret_cast<uintptr_t>(xs) & 15) == 0 && (reinterpret_cast<uintptr_t>(ds) & 15) == 0)
                           ? 4 * groups
                           : 0;
    const size_t smem = kDispBarBytes + (size_t)warps * stages * (chunk + sbytes);
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<capped_grid(units, warps, sms, 1), warps * 32, smem, stream>>>(
        rt, nch, stages, chunk, static_cast<const uint8_t*>(x), xs, static_cast<uint8_t*>(dst), ds, row_bytes, groups,
        sbytes);
    return cudaGetLastError();
}

template <int ACC, class Route, int U = kChainU, int KB = kChainKB>
cudaError_t launch_combine_chain_vec(const Route& rt, long long max_units, int nvec, const void* y, void* out,
                                     const MoveShape& sh, cudaStream_t stream, float* acc) {
    const int nspan = (nvec + 32 * U - 1) / (32 * U);
    const long long units = max_units * nspan;
    if (units == 0) return cudaSuccess;
    auto kern = combine_chain_vec_kernel<ACC, U, KB, Route>;
    const int occ = blocks_per_sm(reinterpret_cast<const void*>(kern), kMoveThreads, 0);
    // like the vector dispatch: several times the resident CTAs unless the
    // tuning sets the combine's SMs or CTAs per SM
    const bool persistent = sh.combine_sms > 0 || sh.combine_ctas > 0;
    const int per_sm = persistent ? (sh.combine_ctas > 0 ? min(sh.combine_ctas, occ) : occ) : occ * kVecOversubscribe;
    const bool acc_v8 = (reinterpret_cast<uintptr_t>(acc) & 31) == 0;
    return launch_pdl(kern, dim3(capped_grid(units, kMoveWarps, mover_sms(sh.combine_sms), per_sm)),
                      dim3(kMoveThreads), 0, stream, rt, nvec, nspan, static_cast<const uint4*>(y),
                      static_cast<uint4*>(out), acc, acc_v8);
}

// Sums at most nl partner rows per unit.  The bulk pipeline's stage holds
// kCombStageBytes: 8 partners x 512 B, or fewer partners with longer pieces
// so that a warp keeps the same bytes in flight; more than 8 partners, or a
// vector combine asked for by the tuning, go to the register kernel.
constexpr int kCombStageBytes = 8 * kCombChunk;

template <class Route>
cudaError_t launch_combine_route(const Route& rt, long long max_units, int nvec, int nl, const void* y, void* out,
                                 const MoveShape& sh, cudaStream_t stream) {
    constexpr int W = kCombWarps, S = kCombStages, B = kCombStageBytes, C = kCombCtasPerSm;
    if (sh.combine_kind != MOE_MOVE_VECTOR) {
        if (nl <= 2) return launch_combine_bulk<W, S, B / 2, 2, false, C, Route>(rt, max_units, nvec, y, out, sh, stream);
        if (nl <= 4) return launch_combine_bulk<W, S, B / 4, 4, false, C, Route>(rt, max_units, nvec, y, out, sh, stream);
        if (nl <= 8) return launch_combine_bulk<W, S, B / 8, 8, false, C, Route>(rt, max_units, nvec, y, out, sh, stream);
    }
    return launch_combine_chain_vec<kAccNone, Route, kFlatVecU, kFlatVecKB>(rt, max_units, nvec, y, out, sh, stream,
                                                                          nullptr);
}

template <int ACC, class Route>
cudaError_t launch_combine_packed(const Route& rt, long long max_units, int nvec, const void* y, void* out,
                                  const MoveShape& sh, cudaStream_t stream, float* acc = nullptr) {
    using Sh = PackedShape<ACC>;
    const int row_bytes = nvec * 16;
    const int nspan = ((row_bytes + kPiece - 1) / kPiece + kPackSlots - 1) / kPackSlots;
    const long long units = max_units * nspan;
    if (units == 0) return cudaSuccess;
    auto kern = combine_packed_kernel<ACC, Route>;
    const size_t smem = (size_t)Sh::kWarps * Sh::kStages * Sh::kStageBytes;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int per_sm = sh.combine_ctas > 0 ? min(sh.combine_ctas, Sh::kCtasPerSm) : Sh::kCtasPerSm;
    const int grid = capped_grid(units, Sh::kWarps, mover_sms(sh.combine_sms), per_sm);
    // Every chain piece starts at a multiple of 1 KB from the row start and a
    // row is 4h bytes (h % 8 == 0), so a 32-byte aligned base aligns them all.
    const bool acc_v8 = (reinterpret_cast<uintptr_t>(acc) & 31) == 0;
    kern<<<grid, Sh::kWarps * 32, smem, stream>>>(rt, static_cast<const uint8_t*>(y), static_cast<uint8_t*>(out),
                                                  row_bytes, acc, acc_v8);
    return cudaGetLastError();
}

// The dispatch kind a route runs when the tuning leaves it to the library.
int dispatch_kind(const MoveShape& sh) {
    return sh.dispatch_kind == MOE_MOVE_BULK ? MOE_MOVE_BULK : MOE_MOVE_VECTOR;
}

long long relay_units_bound(const MoveArgs& m, const RelayArgs& r) {
    const long long most = (long long)m.T * (m.k < r.H ? m.k : r.H);
    return most < r.cap ? most : r.cap;
}

}  // namespace

cudaError_t launch_dispatch(const MoveArgs& m, const void* x, const float* xs, void* recv,
                            float* rs, int groups, cudaStream_t stream) {
    const SlotRoute rt{m.pos, nullptr, m.T, m.k, m.T * m.k};
    return launch_dispatch_route<SlotRoute, false>(rt, m.T, m.nvec * 16, x, xs, recv, rs, groups, m.shape,
                                                   dispatch_kind(m.shape), false, stream);
}

cudaError_t launch_combine(const MoveArgs& m, const void* y, const float* w, void* out,
                           cudaStream_t stream) {
    const SlotRoute rt{m.pos, w, m.T, m.k, m.T * m.k};
    return launch_combine_route(rt, m.T, m.nvec, m.k, y, out, m.shape, stream);
}

cudaError_t launch_dispatch_group(const MoveArgs& m, const GroupArgs& ga, const void* x, const float* xs, void* recv,
                                  float* rs, int groups, cudaStream_t stream) {
    const GroupSlotRoute rt{m.pos, nullptr, ga.ids, ga.group, ga.g, m.T, m.k, ga.E, m.T * m.k};
    return launch_dispatch_route<GroupSlotRoute, true>(rt, m.T, m.nvec * 16, x, xs, recv, rs, groups, m.shape,
                                                       dispatch_kind(m.shape), true, stream);
}

cudaError_t launch_combine_group(const MoveArgs& m, const GroupArgs& ga, const void* y, const float* w, float* acc,
                                 void* out, cudaStream_t stream) {
    const GroupSlotRoute rt{m.pos, w, ga.ids, ga.group, ga.g, m.T, m.k, ga.E, m.T * m.k};
    const MoveShape& sh = m.shape;
    if (ga.G == 1) return launch_combine_route(rt, m.T, m.nvec, m.k, y, out, sh, stream);
    if (m.k <= kPackSlots && sh.combine_kind == MOE_MOVE_BULK) {
        // the shared-memory pipeline, packed: a group holds about k / G of a token's slots
        if (ga.g == 0) return launch_combine_packed<kAccFirst>(rt, m.T, m.nvec, y, out, sh, stream, acc);
        if (ga.g == ga.G - 1) return launch_combine_packed<kAccLast>(rt, m.T, m.nvec, y, out, sh, stream, acc);
        return launch_combine_packed<kAccMid>(rt, m.T, m.nvec, y, out, sh, stream, acc);
    }
    // By default the chain goes through registers: at G = 4 on the prefill-fp8
    // workload the four group combines took 699 us against 870 us for the
    // packed pipeline (decode-EP32-r8: 201 against 286 us).
    if (ga.g == 0) return launch_combine_chain_vec<kAccFirst>(rt, m.T, m.nvec, y, out, sh, stream, acc);
    if (ga.g == ga.G - 1) return launch_combine_chain_vec<kAccLast>(rt, m.T, m.nvec, y, out, sh, stream, acc);
    return launch_combine_chain_vec<kAccMid>(rt, m.T, m.nvec, y, out, sh, stream, acc);
}

cudaError_t launch_relay_dispatch(const MoveArgs& m, const RelayArgs& r, const void* x, const float* xs, void* relay,
                                  float* relay_s, void* recv, float* recv_s, int groups, cudaStream_t stream) {
    const int kind = dispatch_kind(m.shape);
    // hop 1: each token to its relay rows, one per host it reaches
    const HostRoute hop1{r.relay_pos, m.T, r.H, r.cap};
    cudaError_t e = launch_dispatch_route<HostRoute, false>(hop1, m.T, m.nvec * 16, x, xs, relay, relay_s, groups,
                                                            m.shape, kind, true, stream);
    if (e != cudaSuccess) return e;
    // hop 2: each relay row to the receive rows of its host's slots
    const RelaySlotRoute hop2{r.relay_src, r.slot_relay, m.pos, nullptr, r.n_relay, m.T, m.k, m.T * m.k, r.cap};
    return launch_dispatch_route<RelaySlotRoute, false>(hop2, relay_units_bound(m, r), m.nvec * 16, relay, relay_s,
                                                        recv, recv_s, groups, m.shape, kind, true, stream);
}

cudaError_t launch_relay_combine(const MoveArgs& m, const RelayArgs& r, const void* y, const float* w, void* partial,
                                 void* out, cudaStream_t stream) {
    const MoveShape& sh = m.shape;
    // hop 1: each token's k expert rows, summed per host into its relay rows
    cudaError_t e;
    if (m.k <= 8 && sh.combine_kind != MOE_MOVE_VECTOR) {
        const TokenRelayRoute hop1{m.pos, w, r.slot_relay, m.T, m.k, m.T * m.k, r.cap};
        e = launch_combine_bulk<kCombWarps, kCombStages, kCombChunk, 8, true, kCombCtasPerSm>(hop1, m.T, m.nvec, y,
                                                                                            partial, sh, stream);
    } else {
        const RelaySlotRoute hop1{r.relay_src, r.slot_relay, m.pos, w, r.n_relay, m.T, m.k, m.T * m.k, r.cap};
        e = launch_combine_route(hop1, relay_units_bound(m, r), m.nvec, m.k, y, partial, sh, stream);
    }
    if (e != cudaSuccess) return e;
    // hop 2: each token sums its relay rows in ascending host order
    const HostRoute hop2{r.relay_pos, m.T, r.H, r.cap};
    return launch_combine_route(hop2, m.T, m.nvec, m.k < r.H ? m.k : r.H, partial, out, sh, stream);
}

cudaError_t launch_dispatch_quant(const MoveArgs& m0, const void* x, void* recv, float* rs, int h,
                                  cudaStream_t stream) {
    MoveArgs m = m0;
    m.nchunks = (h + kQuantSpanCols - 1) / kQuantSpanCols;  // spans per row
    const long long units = (long long)m.T * m.nchunks;
    if (units == 0) return cudaSuccess;
    // 32-byte pieces where both row arrays allow them (rows are multiples of
    // 256 bytes of input and 128 of codes), else 16-byte ones
    const bool v32 = (reinterpret_cast<uintptr_t>(x) & 31) == 0 && (reinterpret_cast<uintptr_t>(recv) & 31) == 0;
    auto kern = v32 ? dispatch_quant_kernel<32> : dispatch_quant_kernel<16>;
    // like the vector dispatch: a grid of several times the resident CTAs
    // (a tuning that sets SMs or CTAs per SM gets a persistent one)
    const MoveShape& sh = m.shape;
    const int occ = blocks_per_sm(reinterpret_cast<const void*>(kern), kMoveThreads, 0);
    const bool persistent = sh.dispatch_sms > 0 || sh.dispatch_ctas > 0;
    const int per_sm = persistent ? (sh.dispatch_ctas > 0 ? min(sh.dispatch_ctas, occ) : occ) : occ * kVecOversubscribe;
    return launch_pdl(kern, dim3(capped_grid(units, kMoveWarps, mover_sms(sh.dispatch_sms), per_sm)),
                      dim3(kMoveThreads), 0, stream, m, static_cast<const uint8_t*>(x), static_cast<uint8_t*>(recv),
                      rs, h);
}

cudaError_t read_move_faults(uint32_t* bits, cudaStream_t stream) {
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_move_faults, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_move_faults, &zero, sizeof(zero), 0,
                                                      cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) *bits = v;
    return e;
}

}  // namespace moe
