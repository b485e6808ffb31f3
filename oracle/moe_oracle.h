/*
 * moe_oracle.h -- the CPU oracle for MoE token layout, dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C++17
 * restatement of what the GPU library computes, written from the problem
 * statement of the pages it follows:
 *   - "Balancing and Beyond: Communication-Centric Optimizations in Expert
 *     Parallelism" (research digest): section 1 (tokens x k x h x 2 B per
 *     layer and direction), section 2 (imbalance ratio = busiest expert over
 *     the layer mean), section 3.2 (Mode 0 / Mode 1 / Mode 2 copies, relay
 *     through the same-index GPU of the remote host, c1 and c2 formulas),
 *     section 3.4 (receive buffers sized batch x k).
 *   - "[GH-ISSUE #250] Profiling when rank unbalance" (tokens each rank
 *     receives from the other hosts and from its own host).
 *   - "Poor HybridEP performance on dual-node 16x B300 GPUs" (rdma_send_bytes
 *     counted once per (token, host); dispatch_with_permute /
 *     combine_with_unpermute round trip).
 * It shares no code, header, table or constant with the CUDA library; only
 * the test suite, the smoke check and the bench's CPU-baseline leg may call
 * it.  Nothing on the product path links it.
 *
 * All arrays are HOST memory, row-major, owned by the caller.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Problem description.  Logical ranks and hosts are index partitions:
 *   rank(e)  = expert_to_rank ? expert_to_rank[e] : e / (E / R)
 *   host(r)  = r / P,   local index li(r) = r % P,   H = R / P
 *   src(t)   = the source rank r in [0, R_src) with
 *              src_offsets[r] <= t < src_offsets[r+1]
 *              (src_offsets == NULL: equal shares of T / R_src tokens). */
typedef struct {
    int32_t T;              /* tokens */
    int32_t h;              /* hidden size (elements per row) */
    int32_t k;              /* top-k slots per token */
    int32_t E;              /* experts */
    int32_t R;              /* logical ranks (destinations) */
    int32_t P;              /* ranks per host */
    int32_t R_src;          /* source ranks; rank r < R_src owns a token range */
    int32_t elem_bytes;     /* 2 = bf16 rows, 1 = fp8 e4m3 rows */
    int32_t scale_group;    /* fp8 only: columns per fp32 scale (128) */
    const int32_t* expert_to_rank;  /* [E] or NULL */
    const int32_t* src_offsets;     /* [R_src + 1] or NULL */
} oracle_problem;

/* Return codes. */
#define ORACLE_OK           0
#define ORACLE_ERR_INVALID  1   /* shapes or placement are inconsistent */
#define ORACLE_ERR_BAD_IDS  2   /* id out of [0, E) or repeated within a row */

/* Layout: counts, exclusive offsets, per-(token, host) mask, positions.
 * Receive order is the stable sort of all T*k slots (t, j) by the key
 * (rank(e), e); within one expert the slots keep ascending t.
 *   expert_count[E], expert_offset[E+1] (expert_offset[E] = T*k),
 *   rank_count[R],   rank_offset[R+1],
 *   host_count[H] = number of tokens with mask[t][H] = 1, host_offset[H+1],
 *   mask[T*H] (u8), pos[T*k], recv_src[T*k] = t*k + j of the slot stored
 *   at each receive row. */
int oracle_layout(const oracle_problem* p, const int32_t* ids,
                  int32_t* expert_count, int32_t* expert_offset,
                  int32_t* rank_count, int32_t* rank_offset,
                  int32_t* host_count, int32_t* host_offset,
                  uint8_t* mask, int32_t* pos, int32_t* recv_src);

/* Statistics by their plain definitions.  Output arrays:
 *   glob[ORACLE_STATS_GLOBAL_WORDS] (see the indices below),
 *   src[9 * R_src]: field-major blocks of R_src words each
 *       tokens, copies, mode0, mode1, mode2,
 *       naive_bytes (= tokens*k*h*2), mode0_bytes, mode1_bytes, mode2_bytes
 *   dst[6 * R]: field-major blocks of R words each
 *       recv_slots, recv_tokens, recv_self, recv_local, recv_remote,
 *       recv_relay
 * The ratio fields of glob are written to ratio[2]:
 *   ratio[0] = max expert count / (T*k/E), ratio[1] = max rank slots / (T*k/R). */
enum {
    ORACLE_G_T = 0, ORACLE_G_SLOTS, ORACLE_G_ROW_BYTES,
    ORACLE_G_MAX_EXPERT, ORACLE_G_ARGMAX_EXPERT, ORACLE_G_MIN_EXPERT,
    ORACLE_G_MAX_RANK_SLOTS, ORACLE_G_MAX_RANK_TOKENS,
    ORACLE_G_SUM_MODE0, ORACLE_G_SUM_MODE1, ORACLE_G_SUM_MODE2,
    ORACLE_G_MAX_SRC_MODE1, ORACLE_G_MAX_SRC_MODE2,
    ORACLE_G_MAX_RECV_REMOTE, ORACLE_G_MAX_RECV_RELAY,
    ORACLE_G_SUM_NAIVE_BYTES, ORACLE_G_SUM_MODE0_BYTES,
    ORACLE_G_SUM_MODE1_BYTES, ORACLE_G_SUM_MODE2_BYTES,
    ORACLE_STATS_GLOBAL_WORDS
};
int oracle_stats(const oracle_problem* p, const int32_t* ids,
                 int64_t* glob, double* ratio, int64_t* src, int64_t* dst);

/* Dispatch: recv[pos[t*k+j]] = x[t] (row bytes h*elem_bytes); for fp8 also
 * recv_scales[pos[t*k+j]] = x_scales[t] (h/scale_group floats). */
void oracle_dispatch(const oracle_problem* p, const int32_t* pos,
                     const uint8_t* x, const float* x_scales,
                     uint8_t* recv, float* recv_scales);

/* Combine: out[t] = bf16_rne(fma chain over j = 0..k-1 ascending, starting
 * from 0.0f, of w[t*k+j] * y[pos[t*k+j]]).  y and out hold bf16 bit patterns. */
void oracle_combine(const oracle_problem* p, const int32_t* pos,
                    const uint16_t* y, const float* w, uint16_t* out);

/* Mode 2 relay ("Balancing and Beyond", section 3.2: one network copy per
 * token and remote host, fanned out there; combine sums on the relay GPU
 * before sending back).  On one buffer:
 *   relay_pos[T*H]: for a token t and host H with mask[t][H] = 1 the relay row
 *     host_offset[H] + #{t' < t : mask[t'][H] = 1}, otherwise -1.
 *   relay dispatch: relay[relay_pos[t][H]] = x[t] (hop 1), then
 *     recv[pos[t, j]] = relay[relay_pos[t][host(e_j)]] (hop 2, the fan-out);
 *     fp8 scales travel with their rows.
 *   relay combine: partial[relay_pos[t][H]] = bf16_rne(fma chain over the
 *     slots j of t on host H in ascending j, from 0.0f, of w[t, j] *
 *     y[pos[t, j]]) (hop 1), then out[t] = bf16_rne(sum over hosts H with the
 *     mask bit in ascending H, from 0.0f, of the fp32 value of the partial)
 *     (hop 2). */
int oracle_relay_layout(const oracle_problem* p, const int32_t* ids, int32_t* relay_pos);
void oracle_relay_dispatch(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                           const int32_t* relay_pos, const uint8_t* x, const float* x_scales,
                           uint8_t* relay, float* relay_scales, uint8_t* recv, float* recv_scales);
void oracle_relay_combine(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                          const int32_t* relay_pos, const uint16_t* y, const float* w,
                          uint16_t* partial, uint16_t* out);

/* Per-expert-group overlap ("Balancing and Beyond", section 3.3 and its
 * Figure 4: the experts are split into G groups, each dispatched, computed
 * and combined in turn, so that a group's combine can overlap the next
 * group's dispatch and every expert weight is loaded once).
 *   expert groups: every rank's experts, in ascending e, are cut into G
 *     contiguous runs: group(e) = floor(li(e) * G / n(rank(e))), li(e) the
 *     index of e among its rank's experts and n(r) their number.
 *   group dispatch g: recv[pos[t, j]] = x[t] for the slots whose expert is in
 *     group g (scales with them); other receive rows are not written.
 *   group combine g of G: one fp32 fma chain per token runs through the groups
 *     in ascending g and, inside a group, the token's slots of that group in
 *     ascending j; group 0 starts it from 0.0f, every other group continues
 *     from acc[t]; groups before the last write the chain to acc[t] (fp32),
 *     the last writes out[t] = bf16_rne(chain). */
int oracle_expert_groups(const oracle_problem* p, int G, int32_t* group);
void oracle_dispatch_group(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                           const int32_t* group, int g, const uint8_t* x, const float* x_scales,
                           uint8_t* recv, float* recv_scales);
void oracle_combine_group(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                          const int32_t* group, int g, int G, const uint16_t* y, const float* w,
                          float* acc, uint16_t* out);

/* Per-step intra-host expert swap ("Balancing and Beyond", section 3.1 and
 * its Figure 2(b)).  Load of rank r: L_r = sum of expert_count over its
 * experts.  In every host the ranks are ordered by load (descending, ties by
 * rank index) and the i-th heaviest is paired with the i-th lightest.  For a
 * pair (a, b) every exchange of one expert x of a with one expert y of b gives
 * max(L_a - c_x + c_y, L_b - c_y + c_x); the exchange with the smallest such
 * maximum is taken (ties: smallest x, then smallest y) and accepted when it
 * lowers the pair's maximum max(L_a, L_b) by at least max(tau, 1) tokens.
 * Outputs: new_expert_to_rank[E] (the placement after the accepted swaps) and
 * swaps[H * (P/2) * 6] = for each host and pair: rank a, rank b, x, y (-1 when
 * a rank has no expert), old max, new max; accepted pairs are those whose
 * x is moved in new_expert_to_rank.  Returns ORACLE_ERR_INVALID for a bad
 * problem. */
int oracle_swap_plan(const oracle_problem* p, const int32_t* expert_count, int32_t tau,
                     int32_t* new_expert_to_rank, int32_t* swaps);

/* Quantise-in-dispatch: for every token row of bf16 x and every group of
 * scale_group columns, scale = amax / 448 (fp32 division; 1 when the group is
 * all zeros) and codes = e4m3(x / scale) (fp32 division, round to nearest
 * even, saturating at +-448); the codes and scales of token t are written to
 * every receive row pos[t*k+j], like oracle_dispatch. */
void oracle_quantize_dispatch(const oracle_problem* p, const int32_t* pos, const uint16_t* x_bf16,
                              uint8_t* recv_codes, float* recv_scales);

/* FP8 E4M3 (OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite 448) written from the format
 * definition: round to nearest even, saturating to +-448 for finite inputs
 * beyond it; NaN maps to 0x7F. */
uint8_t oracle_f32_to_e4m3_sat(float f);
float oracle_e4m3_to_f32(uint8_t c);

/* bf16 helpers written from the bfloat16 format (the upper 16 bits of an
 * IEEE-754 binary32) and IEEE round-to-nearest-even; exported so the tests
 * can pin them against a library conversion. */
uint16_t oracle_f32_to_bf16_rne(float f);
float oracle_bf16_to_f32(uint16_t b);

#ifdef __cplusplus
}
#endif
#endif
