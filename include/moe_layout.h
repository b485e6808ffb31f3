/*
 * moe_layout.h -- C-ABI of the GB300 (sm_103a) MoE token layout, dispatch
 * and combine library (libmoe_layout.so).
 *
 * What it computes.  The expert-parallel all-to-all of an MoE layer sends each
 * token to its top-k experts and brings the k expert outputs back as a
 * gate-weighted sum ("Balancing and Beyond: Communication-Centric
 * Optimizations in Expert Parallelism", section 1; the HybridEP issue "Poor
 * HybridEP performance on dual-node 16x B300 GPUs" names the single-GPU halves
 * dispatch_with_permute and combine_with_unpermute).  Here the logical EP
 * ranks and hosts are partitions of one GPU's memory:
 *
 *   rank(e) = expert_to_rank ? expert_to_rank[e] : e / (E / R)
 *   host(r) = r / P,  local index li(r) = r % P,  H = R / P
 *   src(t)  = source rank of token t (tokens split over ranks 0..R_src-1)
 *
 * Call order per MoE layer: moe_layout -> (moe_stats) -> moe_dispatch ->
 * [experts] -> moe_combine.  All calls are asynchronous on the given stream;
 * only moe_stats, moe_status, moe_move_faults and moe_selftest_bounded_waits
 * synchronise it.  Every entry
 * point opens an NVTX range of its own name (header-only NVTX 3: free when no
 * profiler is attached).
 *
 * Memory.  The caller allocates every buffer (device memory unless stated)
 * and the workspace; the library allocates nothing and never frees.  It keeps
 * no state between calls, with one exception: moe_layout_noalloc's fixed
 * scratch array (see there), which every call of that entry point shares.
 * Inputs must stay valid until the stream has run the work.  A workspace may
 * be reused by later calls on the same stream; two calls that may run
 * concurrently need two workspaces.
 *
 * Errors.  Every entry point returns a moe_status code.  Arguments that the
 * host can check (sizes, NULL or misaligned pointers) are rejected before any
 * work is enqueued.  Data-dependent faults found on the device (an expert id
 * out of [0, E), an id repeated within a token, a placement entry out of
 * [0, R), bad source offsets) never fault the GPU: they set bits of a status
 * word in the workspace, the affected slot is placed as if it were expert 0 so
 * that every write stays in bounds, and moe_status reports them.
 */
#ifndef MOE_LAYOUT_H
#define MOE_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,   /* bad sizes, NULL pointers, bad placement/offsets */
    MOE_ERR_CUDA = 2,      /* a CUDA launch or copy failed */
    MOE_ERR_BAD_IDS = 3,   /* an expert id out of [0, E) or repeated in a row */
    MOE_ERR_ALIGN = 4,     /* a row buffer is not 16-byte aligned */
    MOE_ERR_CAPACITY = 5,  /* the problem needs more scratch than
                              moe_layout_noalloc's fixed buffer holds, or
                              more relay rows than moe_relay_t holds */
    MOE_ERR_TIMEOUT = 6    /* a bounded device wait gave up (see
                              MOE_STATUS_TIMEOUT); outputs are incomplete */
} moe_status_code;

typedef enum {
    MOE_DTYPE_BF16 = 0,      /* rows of h bf16 values */
    MOE_DTYPE_FP8_E4M3 = 1   /* rows of h e4m3 bytes + h/128 fp32 scales */
} moe_dtype;

/* Device status-word bits reported by moe_status. */
#define MOE_STATUS_ID_RANGE   0x1u   /* id < 0 or id >= E */
#define MOE_STATUS_ID_REPEAT  0x2u   /* the same id twice in one token */
#define MOE_STATUS_PLACEMENT  0x4u   /* expert_to_rank[e] outside [0, R) */
#define MOE_STATUS_SRC_OFFSET 0x8u   /* src_rank_offsets not ascending 0..T */
#define MOE_STATUS_TIMEOUT    0x10u  /* the layout's grid barrier waited more
                                        than one second and gave up */
#define MOE_STATUS_RELAY_CAPACITY 0x20u  /* moe_relay_layout: the layout has
                                        more relay rows than moe_relay_t's
                                        capacity (rows past it are dropped) */

/* Limits checked on the host. */
#define MOE_MAX_TOPK     32
#define MOE_MAX_EXPERTS  1024
#define MOE_MAX_RANKS    1024
#define MOE_MAX_HOSTS    64
#define MOE_MAX_HIDDEN   (1 << 20)  /* columns of a row: row bytes stay far inside int32 */
#define MOE_FP8_GROUP    128   /* columns per fp32 scale */

/* Launch shapes of the layout and the row movers.  The pages' HybridEP issue lists the
 * knobs of that library ("Poor HybridEP performance on dual-node 16x B300
 * GPUs": NUM_OF_TOKENS_PER_CHUNK_*, NUM_SMS_DISPATCH / NUM_SMS_COMBINE,
 * NUM_BLOCKS_PERMUTE / NUM_BLOCKS_UNPERMUTE); these are their counterparts on
 * one GPU.  Any field left 0 keeps the library's default; the shapes change
 * speed only, never a byte of the results.  Out-of-range values give
 * MOE_ERR_INVALID before anything is enqueued.
 *   dispatch_kind: MOE_MOVE_AUTO (default), MOE_MOVE_VECTOR (rows through
 *     registers with 32- or 16-byte vector loads and stores) or MOE_MOVE_BULK
 *     (rows through shared memory with bulk copies, cp.async.bulk).
 *   dispatch_sms / combine_sms: SMs the mover's grid covers, 1 .. the GPU's
 *     SM count (fewer leave SMs to work that overlaps the mover).
 *   dispatch_ctas_per_sm: vector dispatch CTAs per SM, 1 .. 8 (capped by
 *     occupancy).
 *   dispatch_warps, dispatch_stages, dispatch_chunk_bytes: bulk dispatch
 *     warps per CTA (1 .. 16), shared-memory stages per warp (1 .. 8) and
 *     bytes of a source row per stage (a multiple of 16, 256 .. 32768); their
 *     product must fit in 220 KB of shared memory.
 *   combine_kind: MOE_MOVE_AUTO (default: bulk for moe_combine and the relay,
 *     vector for the expert-group chain of moe_combine_group), MOE_MOVE_BULK
 *     (partner pieces gathered into shared memory by bulk copies; at most 8
 *     partners, more fall back to vector) or MOE_MOVE_VECTOR (rows through
 *     registers with vector loads).
 *   combine_ctas_per_sm: bulk combine CTAs per SM, 1 .. 3.
 *   layout_kind: the form of moe_layout's kernels.  MOE_LAYOUT_AUTO (default:
 *     the first of the three below whose grid fits on the GPU at once),
 *     MOE_LAYOUT_SPLIT (one cooperative kernel whose position blocks wait only
 *     for the expert histograms, while separate blocks count tokens per rank
 *     and host for the statistics; B blocks of 128 tokens, B more that count
 *     them, and 2 that write counts, offsets and statistics),
 *     MOE_LAYOUT_FUSED (one cooperative kernel, each block counting and then
 *     ranking its tokens; B + 1 blocks) or MOE_LAYOUT_TWO_KERNELS (a counting
 *     kernel, then a ranking kernel; any T).  A form whose grid does not fit
 *     gives way to the next one. */
#define MOE_MOVE_AUTO   0
#define MOE_MOVE_VECTOR 1
#define MOE_MOVE_BULK   2
#define MOE_LAYOUT_AUTO        0
#define MOE_LAYOUT_SPLIT       1
#define MOE_LAYOUT_FUSED       2
#define MOE_LAYOUT_TWO_KERNELS 3
typedef struct moe_tuning {
    int32_t dispatch_kind;
    int32_t dispatch_sms;
    int32_t dispatch_ctas_per_sm;
    int32_t dispatch_warps;
    int32_t dispatch_stages;
    int32_t dispatch_chunk_bytes;
    int32_t combine_kind;
    int32_t combine_sms;
    int32_t combine_ctas_per_sm;
    int32_t layout_kind;
    int32_t reserved[6];          /* must be 0 */
} moe_tuning;

/* The problem, fixed for one layer.  Sizes:
 *   num_tokens T >= 0, hidden h in [1, 2^20] (bf16: h % 8 == 0; fp8: h % 128 == 0),
 *   topk k in [1, 32], num_experts E in [1, 1024], num_ranks R in [1, 1024],
 *   ranks_per_host P with R % P == 0 and R / P <= 64,
 *   num_src_ranks R_src in [1, R], T * k < 2^31.
 * expert_to_rank: device int32 [E] or NULL (then E % R == 0, contiguous
 *   blocks of E/R experts per rank).
 * src_rank_offsets: device int32 [R_src + 1], ascending, 0 .. T, or NULL
 *   (then T % R_src == 0 and each source rank owns T / R_src tokens).
 * tuning: host moe_tuning or NULL (the defaults); read during each call only. */
typedef struct moe_problem {
    int32_t num_tokens;
    int32_t hidden;
    int32_t topk;
    int32_t num_experts;
    int32_t num_ranks;
    int32_t ranks_per_host;
    int32_t num_src_ranks;
    int32_t dtype;                      /* moe_dtype */
    const int32_t* expert_to_rank;      /* device [E] or NULL */
    const int32_t* src_rank_offsets;    /* device [R_src + 1] or NULL */
    const moe_tuning* tuning;           /* host, or NULL for the defaults */
} moe_problem;

/* Layout outputs, all caller-allocated device arrays (int32 unless noted).
 * Receive order: the T*k slots (t, j) stably sorted by (rank(e), e), so each
 * rank's rows and, inside it, each expert's rows are contiguous and an
 * expert's rows keep ascending token order. */
typedef struct moe_layout_t {
    int32_t* expert_count;   /* [E]   slots routed to expert e */
    int32_t* expert_offset;  /* [E+1] first receive row of expert e; [E] = T*k */
    int32_t* rank_count;     /* [R]   slots received by rank r */
    int32_t* rank_offset;    /* [R+1] exclusive scan of rank_count */
    int32_t* host_count;     /* [H]   tokens with host_mask[t][H] = 1 (one
                                      network copy per token and host) */
    int32_t* host_offset;    /* [H+1] exclusive scan of host_count */
    uint8_t* host_mask;      /* [T, H] u8: 1 iff some slot of t goes to host H */
    int32_t* pos;            /* [T, k] receive row of slot (t, j) */
    int32_t* recv_src;       /* [T*k]  t*k + j of the slot held by each row */
    int64_t* stats;          /* optional [moe_stats_words()] int64: when not
                                NULL, moe_layout also computes the statistics
                                record and writes it here (blocks of the
                                layout kernel beside those that write
                                positions; the kernel ends when the record
                                is written); when NULL, the layout
                                skips it and moe_stats_device / moe_stats
                                compute it later from the workspace */
} moe_layout_t;

/* Bytes of workspace needed for a problem ("Balancing and Beyond" section
 * 3.4 sizes receive buffers batch x k; the workspace holds only counters and
 * per-block tables, a few hundred KB at T = 16384).  Returns MOE_ERR_INVALID
 * for a bad problem. */
int moe_workspace_bytes(const moe_problem* problem, size_t* bytes);

/* Layout (counts, exclusive offsets, per-(token, host) de-duplication mask,
 * stable receive positions and their inverse) of the routing ids.
 *   ids: device int32 [T, k], k distinct experts per token
 *        ("Balancing and Beyond" section 3.2: k distinct experts).
 *   workspace: device, moe_workspace_bytes() bytes, 256-byte aligned; it also
 *        keeps the counters the statistics record is made from, until the
 *        next moe_layout with it.
 * The mask implements Mode 2 de-redundancy (section 3.2): one copy per token
 * and host, relayed through the same-index GPU of that host. */
int moe_layout(const moe_problem* problem, const int32_t* ids, void* workspace,
               const moe_layout_t* layout, moe_stream_t stream);

/* Words (int64) of the statistics record of a problem:
 * MOE_STATS_HEADER_WORDS + 9 * R_src + 6 * R. */
size_t moe_stats_words(const moe_problem* problem);

/* The statistics record of a layout: int64 words, moe_stats_words() of them.
 * Header word indices are MOE_ST_*; the two ratios are IEEE doubles stored in
 * int64 words.  Then nine per-source-rank blocks of R_src words
 * (MOE_SRC_*), then six per-destination-rank blocks of R words (MOE_DST_*).
 * Definitions ("Balancing and Beyond": section 2 imbalance ratio = busiest
 * expert over the layer mean; section 3.2 and Panel 1: Mode 0 sends every copy
 * that leaves the GPU, Mode 1 one network copy per expert on another host,
 * Mode 2 one network copy per other host holding any of the token's experts;
 * section 1: tokens x k x h x 2 B; "Profiling when rank unbalance": tokens a
 * rank receives from its own host and from the others):
 *   row bytes rho = 2h (bf16) or h + 4h/128 (fp8 payload + scales);
 *   src_modeX_bytes = src_modeX * rho; src_naive_bytes = tokens * k * h * 2;
 *   recv_self / recv_local / recv_remote = slots rank r receives from itself /
 *   from other ranks of its host / from other hosts; recv_relay = Mode 2
 *   network copies landing on r as the same-index relay GPU. */
#define MOE_STATS_HEADER_WORDS 32
enum {
    MOE_ST_STATUS = 0,          /* device status bits (MOE_STATUS_*) */
    MOE_ST_TOKENS,              /* T */
    MOE_ST_SLOTS,               /* T*k */
    MOE_ST_ROW_BYTES,           /* rho */
    MOE_ST_MAX_EXPERT,          /* max_e expert_count */
    MOE_ST_ARGMAX_EXPERT,       /* smallest e attaining the max */
    MOE_ST_MIN_EXPERT,          /* min_e expert_count */
    MOE_ST_MAX_RANK_SLOTS,      /* max_r rank_count */
    MOE_ST_MAX_RANK_TOKENS,     /* max_r distinct tokens received */
    MOE_ST_SUM_MODE0,           /* sum over source ranks of Mode 0 copies */
    MOE_ST_SUM_MODE1,
    MOE_ST_SUM_MODE2,
    MOE_ST_MAX_SRC_MODE1,       /* straggler view: busiest sender */
    MOE_ST_MAX_SRC_MODE2,
    MOE_ST_MAX_RECV_REMOTE,     /* busiest network receiver, Mode 1 */
    MOE_ST_MAX_RECV_RELAY,      /* busiest network receiver, Mode 2 */
    MOE_ST_SUM_NAIVE_BYTES,
    MOE_ST_SUM_MODE0_BYTES,
    MOE_ST_SUM_MODE1_BYTES,
    MOE_ST_SUM_MODE2_BYTES,
    MOE_ST_IMBALANCE_RATIO,     /* double: max expert count / (T*k/E) */
    MOE_ST_RANK_IMBALANCE,      /* double: max rank slots / (T*k/R) */
    MOE_ST_NUM_HOSTS            /* H; stays the last named word: the words
                                   after it are unused and read 0 */
};
enum { MOE_SRC_TOKENS = 0, MOE_SRC_COPIES, MOE_SRC_MODE0, MOE_SRC_MODE1, MOE_SRC_MODE2,
       MOE_SRC_NAIVE_BYTES, MOE_SRC_MODE0_BYTES, MOE_SRC_MODE1_BYTES, MOE_SRC_MODE2_BYTES,
       MOE_SRC_FIELDS };
enum { MOE_DST_SLOTS = 0, MOE_DST_TOKENS, MOE_DST_SELF, MOE_DST_LOCAL, MOE_DST_REMOTE,
       MOE_DST_RELAY, MOE_DST_FIELDS };

/* Statistics of a layout, copied to HOST memory; synchronises the stream.
 * The quantities are those of "Balancing and Beyond", sections 1 (bytes that
 * leave each rank: tokens x k x h x 2 B) and 2 (imbalance ratio), with the
 * Mode 0/1/2 copy counts of section 3.2; the record format is above.
 *   layout: the layout made by moe_layout.
 *   workspace: the workspace that moe_layout used: the record is computed
 *     from the counters it holds (one small kernel), then copied.  Or NULL
 *     (a moe_layout_noalloc caller has none): the record is copied from
 *     layout->stats, which must then have been set for the layout call.
 *   host_stats: host int64 [moe_stats_words()] (pageable or pinned).
 * Returns, after the copy, what moe_status would return for the record's
 * status word (MOE_ST_STATUS): MOE_OK, MOE_ERR_BAD_IDS, MOE_ERR_INVALID,
 * MOE_ERR_CAPACITY or MOE_ERR_TIMEOUT; MOE_ERR_CUDA when the copy fails.  The
 * record is written to host_stats in every case but MOE_ERR_CUDA.  Not for
 * use inside a stream capture (it synchronises): capture moe_stats_device. */
int moe_stats(const moe_problem* problem, const moe_layout_t* layout,
              const void* workspace, int64_t* host_stats, moe_stream_t stream);

/* The record of "Balancing and Beyond", sections 1 and 2, as for moe_stats,
 * computed on the device, asynchronously (one block on the stream; it can be
 * captured in a CUDA graph), from the counters the last moe_layout with this
 * workspace left there.  It reads nothing that moe_dispatch or moe_combine
 * write, so with layout->stats left NULL a caller can run it on a second
 * stream beside them, off the dispatch's critical path (the layout kernel
 * then ends when the positions are written); it must finish before the
 * workspace's next moe_layout.
 *   workspace: the workspace of the moe_layout call; device_stats: device
 *   int64 [moe_stats_words()], 8-byte aligned. */
int moe_stats_device(const moe_problem* problem, const void* workspace, int64_t* device_stats,
                     moe_stream_t stream);

/* Dispatch-permute: for every slot, recv[pos[t, j]] = x[t] (a byte-exact row
 * copy); for fp8 also recv_scales[pos[t, j]] = x_scales[t].  This is the
 * dispatch of "Balancing and Beyond", section 1 (each token to its top-k
 * experts, one row per chosen expert), with the receive rows expert-contiguous
 * as the permute half of "Poor HybridEP performance on dual-node 16x B300
 * GPUs" (dispatch_with_permute) leaves them; FP8 rows travel with their
 * scales as in that page's FP8 run.
 *   x: [T, h] bf16 or e4m3 bytes; x_scales: fp32 [T, h/128] (fp8) or NULL;
 *   recv: [T*k, h]; recv_scales: fp32 [T*k, h/128] (fp8) or NULL.
 * x and recv must be 16-byte aligned (MOE_ERR_ALIGN otherwise); scale arrays
 * 4-byte aligned.  Only pos is read from the layout. */
int moe_dispatch(const moe_problem* problem, const moe_layout_t* layout,
                 const void* x, const float* x_scales,
                 void* recv, float* recv_scales, moe_stream_t stream);

/* Quantise-in-dispatch: dispatch of bf16 rows that converts them to FP8 on
 * the way ("Balancing and Beyond", section 3.1: the dispatch kernel does the
 * BF16-to-FP8 conversion).  For every token t and every group of 128 columns:
 *   scale = amax / 448 over the group's |x| (fp32 division; 1 when all zero),
 *   code  = e4m3(x / scale) (fp32 division, round to nearest even, saturated
 *           at +-448; OCP 8-bit floating point E4M3),
 * and recv[pos[t, j]] = codes, recv_scales[pos[t, j]] = scales for every j.
 *   problem->dtype must be MOE_DTYPE_FP8_E4M3 (h % 128 == 0);
 *   x_bf16: [T, h] bf16; recv: [T*k, h] e4m3 bytes; recv_scales: fp32
 *   [T*k, h/128].  x_bf16 and recv 16-byte aligned, recv_scales 4-byte.
 * Only pos is read from the layout. */
int moe_dispatch_quant(const moe_problem* problem, const moe_layout_t* layout,
                       const void* x_bf16, void* recv, float* recv_scales, moe_stream_t stream);

/* Combine-unpermute: out[t] = bf16_rne(sum over j = 0..k-1, in ascending j,
 * of w[t, j] * y[pos[t, j]]) with one fp32 fma per term starting from 0.0f.
 * This is the combine of "Balancing and Beyond", section 1 (the k expert
 * outputs of a token brought back as their gate-weighted sum) and the
 * unpermute half of "Poor HybridEP performance on dual-node 16x B300 GPUs"
 * (combine_with_unpermute); the fixed slot order makes it deterministic.
 *   y: bf16 [T*k, h] expert outputs in receive order; weights: fp32 [T, k];
 *   out: bf16 [T, h].  y and out 16-byte aligned.  Only pos is read from the
 * layout. */
int moe_combine(const moe_problem* problem, const moe_layout_t* layout,
                const void* y, const float* weights, void* out, moe_stream_t stream);

/* ---- Mode 2 relay on one buffer ------------------------------------------
 * The hierarchical path of "Balancing and Beyond", section 3.2 (and the
 * "Mode 2" accounting of "Poor HybridEP performance on dual-node 16x B300
 * GPUs"): a token crosses to each remote host it needs once, to the GPU of
 * its own index there, which fans it out to the expert rows on that host; on
 * the way back that GPU sums the host's weighted expert outputs for the token
 * first, so one row per (token, host) crosses again.  On one GPU both hops
 * run through a relay buffer with one row per (token, host) of the layout's
 * host_mask: the token's own host included, so that every slot takes the same
 * two hops.
 *
 * Relay rows (caller-allocated device int32 arrays):
 *   relay_pos[t][H] = host_offset[H] + #{t' < t : host_mask[t'][H] = 1} when
 *                     host_mask[t][H] = 1, else -1        [T, H]
 *   relay_src[r]    = the token of relay row r             [capacity]
 *   slot_relay[t*k + j] = relay_pos[t][host of slot (t, j)]  [T * k]
 * Relay row count = host_offset[H] (the Mode 2 network copies plus one local
 * copy per token whose experts include its own host) <= T * min(k, H). */
typedef struct moe_relay_t {
    int32_t* relay_pos;
    int32_t* relay_src;
    int32_t* slot_relay;
    int64_t capacity;   /* rows the relay buffers hold; T * min(k, H) always fits */
} moe_relay_t;

/* Relay rows of a layout made by moe_layout with this workspace: the
 * per-(token, host) copies of "Balancing and Beyond", section 3.2 (Figure 3:
 * one copy per token and remote host, relayed by the same-index GPU).  Reads the
 * layout's host_mask, host_offset, rank_offset and pos.  Sets
 * MOE_STATUS_RELAY_CAPACITY in the workspace's status word when host_offset[H]
 * exceeds capacity (moe_status then returns MOE_ERR_CAPACITY).  All arrays
 * 4-byte aligned, the workspace 256-byte aligned. */
int moe_relay_layout(const moe_problem* problem, const moe_layout_t* layout, void* workspace,
                     const moe_relay_t* relay, moe_stream_t stream);

/* Two-hop dispatch of "Balancing and Beyond", section 3.2 (Figure 3): the
 * token crosses to each host once, then fans out there.
 * relay[relay_pos[t][H]] = x[t] for every (t, H) with the
 * mask bit (hop 1), then recv[pos[t, j]] = relay[slot_relay[t*k + j]] for every
 * slot (hop 2); fp8 scales travel with their rows.  recv equals what
 * moe_dispatch writes, byte for byte.
 *   relay_rows: [capacity, h] bf16 or e4m3; relay_scales: fp32
 *   [capacity, h/128] (fp8) or NULL; the rest as for moe_dispatch.  Row
 *   buffers 16-byte aligned. */
int moe_dispatch_relay(const moe_problem* problem, const moe_layout_t* layout, const moe_relay_t* relay,
                       const void* x, const float* x_scales, void* relay_rows, float* relay_scales,
                       void* recv, float* recv_scales, moe_stream_t stream);

/* Two-hop combine of "Balancing and Beyond", section 3.2 (Figure 3): the
 * relay GPU sums its host's expert outputs for a token before the way back.
 * bf16 in and out:
 *   hop 1: partial[r] = bf16_rne(sum over the slots j of token t = relay_src[r]
 *          with slot_relay[t*k + j] = r, in ascending j, of w[t, j] *
 *          y[pos[t, j]]), one fp32 fma per term from 0.0f;
 *   hop 2: out[t] = bf16_rne(sum over the hosts H with host_mask[t][H] = 1, in
 *          ascending H, of partial[relay_pos[t][H]]), fp32 adds from 0.0f.
 * With one host this equals moe_combine bit for bit; otherwise it differs
 * from it by the rounding of the partials to bf16.
 *   partial: bf16 [capacity, h]; y, weights, out as for moe_combine. */
int moe_combine_relay(const moe_problem* problem, const moe_layout_t* layout, const moe_relay_t* relay,
                      const void* y, const float* weights, void* partial, void* out, moe_stream_t stream);

/* ---- Per-expert-group calls ----------------------------------------------
 * Per-expert overlap ("Balancing and Beyond", section 3.3 and Figure 4): the
 * experts are split into G groups (2 or 4 on the page); each group is
 * dispatched, computed and combined in turn, so one group's combine can run
 * while the next group's dispatch does, and each expert's weights load once.
 * A caller issues, per group g = 0 .. G-1, moe_dispatch_group, its expert
 * computation and moe_combine_group, on streams of its choice.
 *
 * Expert groups: every rank's experts, in ascending order, are cut into G
 * contiguous runs: group(e) = floor(li(e) * G / n(rank(e))), li(e) the index
 * of e among its rank's experts and n(r) their number (placement of
 * `problem`).  The page does not say how experts are grouped; this gives
 * every rank work in every group.
 *   expert_group: device int32 [E]; num_groups in [1, MOE_MAX_GROUPS]. */
#define MOE_MAX_GROUPS 64
int moe_expert_groups(const moe_problem* problem, int32_t num_groups, int32_t* expert_group,
                      moe_stream_t stream);

/* Dispatch of one expert group ("Balancing and Beyond", section 3.3 and
 * Figure 4: per-expert overlap).  recv[pos[t, j]] = x[t] (scales with it) for
 * the slots whose expert ids[t, j] has expert_group = group; no other receive
 * row is written.  The G groups together write what moe_dispatch writes.
 *   ids: the [T, k] ids the layout was made from; other arguments as for
 *   moe_dispatch. */
int moe_dispatch_group(const moe_problem* problem, const moe_layout_t* layout, const int32_t* ids,
                       const int32_t* expert_group, int32_t group, const void* x, const float* x_scales,
                       void* recv, float* recv_scales, moe_stream_t stream);

/* Combine of one expert group ("Balancing and Beyond", section 3.3 and
 * Figure 4: a group's combine runs while the next group's dispatch does).
 * One fp32 fma chain per token runs through the
 * groups in ascending order and, inside a group, through the token's slots of
 * that group in ascending j: group 0 starts it from 0.0f; every later group
 * continues it from acc[t]; every group but the last stores it to acc[t]
 * (fp32), the last writes out[t] = bf16_rne(chain).  The groups must run in
 * order.  With one group this is moe_combine.
 *   acc: device fp32 [T, h], 16-byte aligned (may be NULL when num_groups is
 *   1); y, weights, out as for moe_combine. */
int moe_combine_group(const moe_problem* problem, const moe_layout_t* layout, const int32_t* ids,
                      const int32_t* expert_group, int32_t group, int32_t num_groups, const void* y,
                      const float* weights, float* acc, void* out, moe_stream_t stream);

/* The pages have no counterpart: the status word is this library's way to
 * report data-dependent faults without faulting the GPU.
 * Waits for the stream, then reads the device status bits of the workspace
 * (the faults found by the last moe_layout and moe_relay_layout).
 * *status_bits receives them; returns MOE_OK, MOE_ERR_BAD_IDS,
 * MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT or MOE_ERR_CUDA. */
int moe_status(const void* workspace, uint32_t* status_bits, moe_stream_t stream);

/* Layout without a caller workspace -- this entry point has no counterpart
 * on the pages; it exists for callers that cannot allocate device memory,
 * such as a plugin inside an inference engine whose device memory the engine
 * plans and owns, or a plain C caller with no device allocator (cudaMalloc
 * also synchronises the device, which a hot path cannot afford).
 *
 * It computes exactly what moe_layout computes, but its scratch is a fixed
 * MOE_NOALLOC_SCRATCH_BYTES array inside the library's own device memory,
 * which every GPU that loads the library holds until the process exits.  It
 * allocates nothing and frees nothing.
 *   - Returns MOE_ERR_CAPACITY, before any work is enqueued, when the
 *     problem's moe_workspace_bytes() exceeds MOE_NOALLOC_SCRATCH_BYTES.  The
 *     workspace grows with T * E (about 4 bytes per expert per 128 tokens,
 *     plus the statistics record), so 2 MiB holds about 245,000 tokens with
 *     E = 256 experts and about 57,000 with E = 1024.
 *   - Each call looks up the array's address on the current device (no
 *     allocation, no synchronisation).  The first call on a device also loads
 *     the library's device code there: make that first call before any stream
 *     capture.
 *   - All calls in the process share the one array per device.  Two calls
 *     that may overlap on the GPU (different streams, or different host
 *     threads) race on it and corrupt each other's layout; serialise them.
 *     Each call clears the counters it needs, so stale contents from an
 *     earlier call do no harm.
 *   - There is no caller workspace, so moe_status cannot read this variant's
 *     device status bits.  They reach the caller through the statistics
 *     record: set layout->stats, and word MOE_ST_STATUS holds the bits (or
 *     call moe_stats with that layout and workspace = NULL).  An id out of
 *     range or repeated still cannot write out of bounds. */
#define MOE_NOALLOC_SCRATCH_BYTES (2u << 20)
int moe_layout_noalloc(const moe_problem* problem, const int32_t* ids,
                       const moe_layout_t* layout, moe_stream_t stream);

/* Per-step intra-host expert swap plan ("Balancing and Beyond", section 3.1
 * and its Figure 2(b)).  Rank loads are the layout's expert_count summed over
 * each rank's experts (the placement of `problem`).  In every host the ranks
 * are ordered by load (descending, ties by rank index) and the i-th heaviest
 * is paired with the i-th lightest; for each pair the one exchange of an
 * expert x of the heavier rank with an expert y of the lighter that gives the
 * smallest pair maximum is chosen (ties: smallest x, then smallest y) and
 * applied when it lowers the pair's maximum by at least max(tau, 1) tokens.
 *   new_expert_to_rank: device int32 [E], the placement after the swaps (pass
 *     it as problem->expert_to_rank of the next step);
 *   swaps: device int32 [H * (ranks_per_host / 2) * 6] or NULL: per host and
 *     pair, rank a, rank b, x, y (-1 if a rank has no expert), old maximum,
 *     best new maximum (the swap was applied when new_expert_to_rank moved x).
 * Needs E <= 1024 (ids fit the search key) like every other call. */
int moe_swap_plan(const moe_problem* problem, const moe_layout_t* layout, int32_t tau,
                  int32_t* new_expert_to_rank, int32_t* swaps, moe_stream_t stream);

/* The pages have no counterpart (bounded waits of this library's movers).
 * Device faults of the row movers since the last call: bit
 * MOE_FAULT_WAIT_TIMEOUT is set when a bulk-copy pipeline of moe_dispatch or
 * moe_combine waited more than one second for its own copies, gave up, drained
 * them and returned (its output is then incomplete).  Waits for the stream,
 * copies the bits to *bits and clears them. */
#define MOE_FAULT_WAIT_TIMEOUT 0x1u
int moe_move_faults(uint32_t* bits, moe_stream_t stream);

/* The pages have no counterpart.
 * Self-test of the library's bounded device waits (the bulk-copy barrier
 * waits of moe_dispatch / moe_combine and the grid barrier of moe_layout):
 * runs them, with a 10 ms limit, on barriers that can never complete and on
 * barriers that do, without faulting or hanging the GPU.  Allocates nothing;
 * waits for the stream.  *bits receives 0xF when every wait behaved: bit 0 an
 * mbarrier wait gave up, bit 1 an mbarrier wait succeeded, bit 2 a grid
 * barrier wait gave up, bit 3 a grid barrier wait succeeded. */
int moe_selftest_bounded_waits(uint32_t* bits, moe_stream_t stream);

/* A short English description of a moe_status_code. */
const char* moe_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif
