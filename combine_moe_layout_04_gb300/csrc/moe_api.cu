// moe_api.cu -- the extern "C" entry points of libmoe_layout.so: argument
// checks on the host, then kernel launches on the caller's stream, each call
// inside an NVTX range of its own name.  The library allocates no memory and
// keeps no state between calls (moe_noalloc.cu's fixed scratch array aside).

#include <cstdint>
#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace {

using moe::WsLayout;

struct Dims {
    int T, h, k, E, R, P, H, Rs;
    bool fp8;
    moe::MoveShape shape;
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Launch shapes of a moe_tuning (NULL: every default), checked on the host.
int check_tuning(const moe_tuning* t, moe::MoveShape* sh) {
    *sh = moe::MoveShape{};
    if (t == nullptr) return MOE_OK;
    auto in = [](int v, int lo, int hi) { return v == 0 || (v >= lo && v <= hi); };
    if (!in(t->dispatch_kind, MOE_MOVE_VECTOR, MOE_MOVE_BULK) || !in(t->combine_kind, MOE_MOVE_VECTOR, MOE_MOVE_BULK))
        return MOE_ERR_INVALID;
    if (!in(t->dispatch_sms, 1, 1 << 16) || !in(t->combine_sms, 1, 1 << 16)) return MOE_ERR_INVALID;
    if (!in(t->dispatch_ctas_per_sm, 1, 8) || !in(t->dispatch_warps, 1, 16) || !in(t->dispatch_stages, 1, 8))
        return MOE_ERR_INVALID;
    if (!in(t->dispatch_chunk_bytes, 256, 32768) || t->dispatch_chunk_bytes % 16 != 0) return MOE_ERR_INVALID;
    if (!in(t->combine_ctas_per_sm, 1, 3)) return MOE_ERR_INVALID;
    if (!in(t->layout_kind, MOE_LAYOUT_SPLIT, MOE_LAYOUT_TWO_KERNELS)) return MOE_ERR_INVALID;
    for (int r : t->reserved)
        if (r != 0) return MOE_ERR_INVALID;
    // the bulk dispatch's stages must fit in shared memory (the larger of the
    // two default warp counts stands in for a field left 0)
    const long long warps = t->dispatch_warps ? t->dispatch_warps : 6;
    const long long stages = t->dispatch_stages ? t->dispatch_stages : 4;
    const long long chunk = t->dispatch_chunk_bytes ? t->dispatch_chunk_bytes : 7168;
    if (warps * stages * chunk > 220 * 1024) return MOE_ERR_INVALID;
    sh->dispatch_kind = t->dispatch_kind;
    sh->dispatch_sms = t->dispatch_sms;
    sh->dispatch_ctas = t->dispatch_ctas_per_sm;
    sh->dispatch_warps = t->dispatch_warps;
    sh->dispatch_stages = t->dispatch_stages;
    sh->dispatch_chunk = t->dispatch_chunk_bytes;
    sh->combine_kind = t->combine_kind;
    sh->combine_sms = t->combine_sms;
    sh->combine_ctas = t->combine_ctas_per_sm;
    sh->layout_kind = t->layout_kind;
    return MOE_OK;
}

int check_problem(const moe_problem* p, Dims* d) {
    if (p == nullptr) return MOE_ERR_INVALID;
    if (check_tuning(p->tuning, &d->shape) != MOE_OK) return MOE_ERR_INVALID;
    d->T = p->num_tokens; d->h = p->hidden; d->k = p->topk; d->E = p->num_experts;
    d->R = p->num_ranks; d->P = p->ranks_per_host; d->Rs = p->num_src_ranks;
    d->fp8 = p->dtype == MOE_DTYPE_FP8_E4M3;
    if (p->dtype != MOE_DTYPE_BF16 && p->dtype != MOE_DTYPE_FP8_E4M3) return MOE_ERR_INVALID;
    if (d->T < 0 || d->h <= 0 || d->h > MOE_MAX_HIDDEN) return MOE_ERR_INVALID;
    if (d->k < 1 || d->k > MOE_MAX_TOPK) return MOE_ERR_INVALID;
    if (d->E < 1 || d->E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID;
    if (d->R < 1 || d->R > MOE_MAX_RANKS || d->P < 1 || d->R % d->P != 0) return MOE_ERR_INVALID;
    d->H = d->R / d->P;
    if (d->H > MOE_MAX_HOSTS) return MOE_ERR_INVALID;
    if (d->Rs < 1 || d->Rs > d->R) return MOE_ERR_INVALID;
    if ((long long)d->T * d->k >= (1LL << 31)) return MOE_ERR_INVALID;
    if (p->expert_to_rank == nullptr && d->E % d->R != 0) return MOE_ERR_INVALID;
    if (p->src_rank_offsets == nullptr && d->T % d->Rs != 0) return MOE_ERR_INVALID;
    if (d->fp8 ? (d->h % MOE_FP8_GROUP != 0) : (d->h % 8 != 0)) return MOE_ERR_INVALID;
    if (!aligned(p->expert_to_rank, 4) || !aligned(p->src_rank_offsets, 4)) return MOE_ERR_ALIGN;
    return MOE_OK;
}

// Arrays sized by T may be NULL when T == 0.
bool layout_complete(const moe_layout_t* l, int T) {
    if (!l || !l->expert_count || !l->expert_offset || !l->rank_count || !l->rank_offset ||
        !l->host_count || !l->host_offset)
        return false;
    return T == 0 || (l->host_mask && l->pos && l->recv_src);
}

// Relay arrays sized by T may be NULL when T == 0; capacity >= 0.
bool relay_complete(const moe_relay_t* r, int T) {
    if (r->capacity < 0) return false;
    return T == 0 || (r->relay_pos && r->slot_relay && (r->relay_src || r->capacity == 0));
}

int relay_cap(const moe_relay_t* r) {
    return r->capacity > (int64_t)INT32_MAX ? INT32_MAX : (int)r->capacity;
}

moe::RelayArgs relay_args(const moe_relay_t* relay, const moe_layout_t* layout, const Dims& d) {
    moe::RelayArgs r{};
    r.relay_pos = relay->relay_pos;
    r.relay_src = relay->relay_src;
    r.slot_relay = relay->slot_relay;
    r.n_relay = layout->host_offset + d.H;
    r.H = d.H;
    r.cap = relay_cap(relay);
    return r;
}

WsLayout ws_layout(const Dims& d) { return moe::make_ws_layout(d.T, d.E, d.R, d.H, d.Rs); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int64_t row_bytes(const Dims& d);

// The layout kernels' arguments for a problem and workspace (ids and outputs
// are the caller's to fill in).
moe::LayoutArgs layout_args(const moe_problem* problem, const Dims& d, const void* workspace) {
    moe::LayoutArgs a{};
    a.expert_to_rank = problem->expert_to_rank;
    a.src_offsets = problem->src_rank_offsets;
    a.T = d.T; a.k = d.k; a.E = d.E; a.R = d.R; a.P = d.P; a.H = d.H; a.Rs = d.Rs;
    a.h = d.h;
    a.row_bytes = row_bytes(d);
    a.ws = static_cast<uint8_t*>(const_cast<void*>(workspace));
    a.wl = ws_layout(d);
    a.kind = d.shape.layout_kind;
    // the layer means T*k/E and T*k/R, each rounded once as the record defines them
    a.mean_expert = (double)((int64_t)d.T * d.k) / (double)d.E;
    a.mean_rank = (double)((int64_t)d.T * d.k) / (double)d.R;
    return a;
}

// The code a set of device status bits stands for (timeouts first).
int code_of_status(uint32_t bits) {
    if (bits & MOE_STATUS_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (bits & (MOE_STATUS_ID_RANGE | MOE_STATUS_ID_REPEAT)) return MOE_ERR_BAD_IDS;
    if (bits & (MOE_STATUS_PLACEMENT | MOE_STATUS_SRC_OFFSET)) return MOE_ERR_INVALID;
    if (bits & MOE_STATUS_RELAY_CAPACITY) return MOE_ERR_CAPACITY;
    return MOE_OK;
}

int64_t row_bytes(const Dims& d) {
    return d.fp8 ? (int64_t)d.h + 4LL * (d.h / MOE_FP8_GROUP) : 2LL * d.h;
}

}  // namespace

extern "C" {

int moe_workspace_bytes(const moe_problem* problem, size_t* bytes) {
    MOE_NVTX("moe_workspace_bytes");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (bytes == nullptr) return MOE_ERR_INVALID;
    *bytes = ws_layout(d).total;
    return MOE_OK;
}

size_t moe_stats_words(const moe_problem* problem) {
    MOE_NVTX("moe_stats_words");
    Dims d;
    if (check_problem(problem, &d) != MOE_OK) return 0;
    return MOE_STATS_HEADER_WORDS + (size_t)MOE_SRC_FIELDS * d.Rs + (size_t)MOE_DST_FIELDS * d.R;
}

int moe_layout(const moe_problem* problem, const int32_t* ids, void* workspace,
               const moe_layout_t* layout, moe_stream_t stream) {
    MOE_NVTX("moe_layout");
    Dims d;
    int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (!layout_complete(layout, d.T) || workspace == nullptr || (d.T > 0 && ids == nullptr))
        return MOE_ERR_INVALID;
    if (!aligned(workspace, 256) || !aligned(ids, 4) || !aligned(layout->stats, 8)) return MOE_ERR_ALIGN;
    moe::LayoutArgs a = layout_args(problem, d, workspace);
    a.ids = ids;
    a.out = *layout;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = cuda_status(cudaMemsetAsync(workspace, 0, a.wl.acc_bytes, s));
    if (rc != MOE_OK) return rc;
    return cuda_status(moe::launch_layout(a, s));
}

int moe_stats(const moe_problem* problem, const moe_layout_t* layout, const void* workspace,
              int64_t* host_stats, moe_stream_t stream) {
    MOE_NVTX("moe_stats");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || host_stats == nullptr) return MOE_ERR_INVALID;
    if (!aligned(host_stats, 8)) return MOE_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const WsLayout wl = ws_layout(d);
    const void* src = nullptr;
    if (workspace != nullptr) {
        // the record, made now from the counters the layout left in the workspace
        if (!aligned(workspace, 256)) return MOE_ERR_ALIGN;
        moe::LayoutArgs a = layout_args(problem, d, workspace);
        if (moe::launch_stats_compute(a, s) != cudaSuccess) return MOE_ERR_CUDA;
        src = static_cast<const uint8_t*>(workspace) + wl.stats;
    } else {
        // no workspace (moe_layout_noalloc): the record the layout wrote itself
        if (layout->stats == nullptr) return MOE_ERR_INVALID;
        if (!aligned(layout->stats, 8)) return MOE_ERR_ALIGN;
        src = layout->stats;
    }
    cudaError_t e = cudaMemcpyAsync(host_stats, src, 8 * wl.stats_words, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return code_of_status(static_cast<uint32_t>(host_stats[MOE_ST_STATUS]));
}

int moe_stats_device(const moe_problem* problem, const void* workspace, int64_t* device_stats,
                     moe_stream_t stream) {
    MOE_NVTX("moe_stats_device");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (workspace == nullptr || device_stats == nullptr) return MOE_ERR_INVALID;
    if (!aligned(workspace, 256) || !aligned(device_stats, 8)) return MOE_ERR_ALIGN;
    moe::LayoutArgs a = layout_args(problem, d, workspace);
    a.out.stats = device_stats;
    return cuda_status(moe::launch_stats_compute(a, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_dispatch(const moe_problem* problem, const moe_layout_t* layout, const void* x,
                 const float* x_scales, void* recv, float* recv_scales, moe_stream_t stream) {
    MOE_NVTX("moe_dispatch");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || x == nullptr || recv == nullptr) return MOE_ERR_INVALID;
    if (d.fp8 && (x_scales == nullptr || recv_scales == nullptr)) return MOE_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(layout->pos, 4)) return MOE_ERR_ALIGN;
    if (d.fp8 && (!aligned(x_scales, 4) || !aligned(recv_scales, 4))) return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = (int)((d.fp8 ? (int64_t)d.h : 2LL * d.h) / 16);
    const int groups = d.fp8 ? d.h / MOE_FP8_GROUP : 0;
    return cuda_status(moe::launch_dispatch(m, x, x_scales, recv, recv_scales, groups,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int moe_dispatch_quant(const moe_problem* problem, const moe_layout_t* layout, const void* x_bf16,
                       void* recv, float* recv_scales, moe_stream_t stream) {
    MOE_NVTX("moe_dispatch_quant");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (!d.fp8 || layout == nullptr) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || x_bf16 == nullptr || recv == nullptr || recv_scales == nullptr)
        return MOE_ERR_INVALID;
    if (!aligned(x_bf16, 16) || !aligned(recv, 16) || !aligned(recv_scales, 4) || !aligned(layout->pos, 4))
        return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    return cuda_status(moe::launch_dispatch_quant(m, x_bf16, recv, recv_scales, d.h,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int moe_combine(const moe_problem* problem, const moe_layout_t* layout, const void* y,
                const float* weights, void* out, moe_stream_t stream) {
    MOE_NVTX("moe_combine");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || y == nullptr || weights == nullptr || out == nullptr) return MOE_ERR_INVALID;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(weights, 4) || !aligned(layout->pos, 4))
        return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = d.h / 8;  // combine is bf16 in and out
    return cuda_status(moe::launch_combine(m, y, weights, out, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_relay_layout(const moe_problem* problem, const moe_layout_t* layout, void* workspace,
                     const moe_relay_t* relay, moe_stream_t stream) {
    MOE_NVTX("moe_relay_layout");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (!layout_complete(layout, d.T) || workspace == nullptr || relay == nullptr || !relay_complete(relay, d.T))
        return MOE_ERR_INVALID;
    if (!aligned(workspace, 256) || !aligned(relay->relay_pos, 4) || !aligned(relay->relay_src, 4) ||
        !aligned(relay->slot_relay, 4))
        return MOE_ERR_ALIGN;
    if (d.T == 0) return MOE_OK;
    const WsLayout wl = ws_layout(d);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    moe::RelayLayoutArgs a{};
    a.host_mask = layout->host_mask;
    a.host_offset = layout->host_offset;
    a.rank_offset = layout->rank_offset;
    a.pos = layout->pos;
    a.relay_pos = relay->relay_pos;
    a.relay_src = relay->relay_src;
    a.slot_relay = relay->slot_relay;
    a.tiles = reinterpret_cast<int32_t*>(ws + wl.relay_tiles);
    a.status = reinterpret_cast<uint32_t*>(ws + wl.status);
    a.T = d.T; a.k = d.k; a.H = d.H; a.P = d.P;
    a.cap = relay_cap(relay);
    return cuda_status(moe::launch_relay_layout(a, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_dispatch_relay(const moe_problem* problem, const moe_layout_t* layout, const moe_relay_t* relay,
                       const void* x, const float* x_scales, void* relay_rows, float* relay_scales,
                       void* recv, float* recv_scales, moe_stream_t stream) {
    MOE_NVTX("moe_dispatch_relay");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || relay == nullptr || !relay_complete(relay, d.T)) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || layout->host_offset == nullptr || x == nullptr || relay_rows == nullptr ||
        recv == nullptr)
        return MOE_ERR_INVALID;
    if (d.fp8 && (x_scales == nullptr || relay_scales == nullptr || recv_scales == nullptr)) return MOE_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(relay_rows, 16) || !aligned(recv, 16) || !aligned(layout->pos, 4) ||
        !aligned(relay->relay_pos, 4) || !aligned(relay->relay_src, 4) || !aligned(relay->slot_relay, 4))
        return MOE_ERR_ALIGN;
    if (d.fp8 && (!aligned(x_scales, 4) || !aligned(relay_scales, 4) || !aligned(recv_scales, 4)))
        return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = (int)((d.fp8 ? (int64_t)d.h : 2LL * d.h) / 16);
    const moe::RelayArgs r = relay_args(relay, layout, d);
    return cuda_status(moe::launch_relay_dispatch(m, r, x, x_scales, relay_rows, relay_scales, recv, recv_scales,
                                                  d.fp8 ? d.h / MOE_FP8_GROUP : 0,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int moe_combine_relay(const moe_problem* problem, const moe_layout_t* layout, const moe_relay_t* relay,
                      const void* y, const float* weights, void* partial, void* out, moe_stream_t stream) {
    MOE_NVTX("moe_combine_relay");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || relay == nullptr || !relay_complete(relay, d.T)) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || layout->host_offset == nullptr || y == nullptr || weights == nullptr ||
        partial == nullptr || out == nullptr)
        return MOE_ERR_INVALID;
    if (!aligned(y, 16) || !aligned(partial, 16) || !aligned(out, 16) || !aligned(weights, 4) ||
        !aligned(layout->pos, 4) || !aligned(relay->relay_pos, 4) || !aligned(relay->relay_src, 4) ||
        !aligned(relay->slot_relay, 4))
        return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = d.h / 8;  // combine is bf16 in and out
    const moe::RelayArgs r = relay_args(relay, layout, d);
    return cuda_status(moe::launch_relay_combine(m, r, y, weights, partial, out,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int moe_expert_groups(const moe_problem* problem, int32_t num_groups, int32_t* expert_group,
                      moe_stream_t stream) {
    MOE_NVTX("moe_expert_groups");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (num_groups < 1 || num_groups > MOE_MAX_GROUPS || expert_group == nullptr) return MOE_ERR_INVALID;
    if (!aligned(expert_group, 4)) return MOE_ERR_ALIGN;
    return cuda_status(moe::launch_expert_groups(problem->expert_to_rank, d.E, d.R, num_groups, expert_group,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int moe_dispatch_group(const moe_problem* problem, const moe_layout_t* layout, const int32_t* ids,
                       const int32_t* expert_group, int32_t group, const void* x, const float* x_scales,
                       void* recv, float* recv_scales, moe_stream_t stream) {
    MOE_NVTX("moe_dispatch_group");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || expert_group == nullptr || group < 0 || group >= MOE_MAX_GROUPS) return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || ids == nullptr || x == nullptr || recv == nullptr) return MOE_ERR_INVALID;
    if (d.fp8 && (x_scales == nullptr || recv_scales == nullptr)) return MOE_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(layout->pos, 4) || !aligned(ids, 4) ||
        !aligned(expert_group, 4))
        return MOE_ERR_ALIGN;
    if (d.fp8 && (!aligned(x_scales, 4) || !aligned(recv_scales, 4))) return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = (int)((d.fp8 ? (int64_t)d.h : 2LL * d.h) / 16);
    const moe::GroupArgs ga{ids, expert_group, group, 0, d.E};
    return cuda_status(moe::launch_dispatch_group(m, ga, x, x_scales, recv, recv_scales,
                                                  d.fp8 ? d.h / MOE_FP8_GROUP : 0,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int moe_combine_group(const moe_problem* problem, const moe_layout_t* layout, const int32_t* ids,
                      const int32_t* expert_group, int32_t group, int32_t num_groups, const void* y,
                      const float* weights, float* acc, void* out, moe_stream_t stream) {
    MOE_NVTX("moe_combine_group");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || expert_group == nullptr || num_groups < 1 || num_groups > MOE_MAX_GROUPS ||
        group < 0 || group >= num_groups)
        return MOE_ERR_INVALID;
    if (d.T == 0) return MOE_OK;
    if (layout->pos == nullptr || ids == nullptr || y == nullptr || weights == nullptr || out == nullptr ||
        (num_groups > 1 && acc == nullptr))
        return MOE_ERR_INVALID;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(acc, 16) || !aligned(weights, 4) ||
        !aligned(layout->pos, 4) || !aligned(ids, 4) || !aligned(expert_group, 4))
        return MOE_ERR_ALIGN;
    moe::MoveArgs m{};
    m.shape = d.shape;
    m.pos = layout->pos;
    m.T = d.T;
    m.k = d.k;
    m.nvec = d.h / 8;  // combine is bf16 in and out
    const moe::GroupArgs ga{ids, expert_group, group, num_groups, d.E};
    return cuda_status(moe::launch_combine_group(m, ga, y, weights, acc, out,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int moe_status(const void* workspace, uint32_t* status_bits, moe_stream_t stream) {
    MOE_NVTX("moe_status");
    if (workspace == nullptr || status_bits == nullptr) return MOE_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    // The status word sits at offset 0 of every workspace.
    cudaError_t e = cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *status_bits = bits;
    return code_of_status(bits);
}

int moe_swap_plan(const moe_problem* problem, const moe_layout_t* layout, int32_t tau,
                  int32_t* new_expert_to_rank, int32_t* swaps, moe_stream_t stream) {
    MOE_NVTX("moe_swap_plan");
    Dims d;
    const int rc = check_problem(problem, &d);
    if (rc != MOE_OK) return rc;
    if (layout == nullptr || layout->expert_count == nullptr || new_expert_to_rank == nullptr)
        return MOE_ERR_INVALID;
    if (!aligned(layout->expert_count, 4) || !aligned(new_expert_to_rank, 4) || !aligned(swaps, 4))
        return MOE_ERR_ALIGN;
    return cuda_status(moe::launch_swap_plan(layout->expert_count, problem->expert_to_rank, d.E, d.R, d.P,
                                             tau, new_expert_to_rank, swaps,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int moe_move_faults(uint32_t* bits, moe_stream_t stream) {
    MOE_NVTX("moe_move_faults");
    if (bits == nullptr) return MOE_ERR_INVALID;
    return cuda_status(moe::read_move_faults(bits, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_selftest_bounded_waits(uint32_t* bits, moe_stream_t stream) {
    MOE_NVTX("moe_selftest_bounded_waits");
    if (bits == nullptr) return MOE_ERR_INVALID;
    return cuda_status(moe::run_wait_selftest(bits, reinterpret_cast<cudaStream_t>(stream)));
}

const char* moe_status_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_BAD_IDS: return "expert id out of range or repeated within a token";
        case MOE_ERR_ALIGN: return "misaligned buffer";
        case MOE_ERR_CAPACITY: return "problem too large for the fixed layout scratch";
        case MOE_ERR_TIMEOUT: return "a bounded device wait gave up";
        default: return "unknown status";
    }
}

}  // extern "C"
