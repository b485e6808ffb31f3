// moe_oracle.cpp -- TEST INFRASTRUCTURE ONLY: plain single-threaded CPU
// definitions of MoE token layout, statistics, dispatch and combine.
//
// Every function below is the textbook definition written out, with no
// blocking, fusion or reordering: loops over (token, slot), one library
// stable sort, memcpy of rows, and an explicit fma chain.  It shares no code
// with the CUDA library.  Build: g++ -std=c++17 -O2 -ffp-contract=off.

#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

struct Placement {
    int32_t E, R, P, H;
    std::vector<int32_t> rank_of_expert;   // rank(e)
};

// Checks the problem and builds rank(e).  Default placement: experts split in
// equal contiguous blocks over the ranks ("Balancing and Beyond" section 3.2
// model: the E experts are spread evenly over the hosts).
bool make_placement(const oracle_problem* p, Placement* pl) {
    if (p->T < 0 || p->k < 1 || p->E < 1 || p->R < 1 || p->P < 1) return false;
    if (p->R % p->P != 0) return false;
    if (p->R_src < 1 || p->R_src > p->R) return false;
    pl->E = p->E; pl->R = p->R; pl->P = p->P; pl->H = p->R / p->P;
    pl->rank_of_expert.assign(p->E, 0);
    if (p->expert_to_rank) {
        for (int e = 0; e < p->E; ++e) {
            if (p->expert_to_rank[e] < 0 || p->expert_to_rank[e] >= p->R) return false;
            pl->rank_of_expert[e] = p->expert_to_rank[e];
        }
    } else {
        if (p->E % p->R != 0) return false;
        const int per = p->E / p->R;
        for (int e = 0; e < p->E; ++e) pl->rank_of_expert[e] = e / per;
    }
    return true;
}

// src(t): the source rank that owns token t.
bool make_sources(const oracle_problem* p, std::vector<int32_t>* src_of_token) {
    src_of_token->assign(p->T, 0);
    if (p->src_offsets) {
        if (p->src_offsets[0] != 0 || p->src_offsets[p->R_src] != p->T) return false;
        for (int r = 0; r < p->R_src; ++r) {
            if (p->src_offsets[r + 1] < p->src_offsets[r]) return false;
            for (int t = p->src_offsets[r]; t < p->src_offsets[r + 1]; ++t) (*src_of_token)[t] = r;
        }
    } else {
        if (p->T % p->R_src != 0) return false;
        const int per = p->T / p->R_src;
        for (int t = 0; t < p->T; ++t) (*src_of_token)[t] = per ? t / per : 0;
    }
    return true;
}

// Top-k ids must be k distinct experts in [0, E): the routing model of
// "Balancing and Beyond", section 3.2 draws distinct experts per token.
bool ids_valid(const oracle_problem* p, const int32_t* ids) {
    for (int t = 0; t < p->T; ++t) {
        for (int j = 0; j < p->k; ++j) {
            const int32_t e = ids[(size_t)t * p->k + j];
            if (e < 0 || e >= p->E) return false;
            for (int i = 0; i < j; ++i)
                if (ids[(size_t)t * p->k + i] == e) return false;
        }
    }
    return true;
}

// mask[t][H] = 1 iff some slot of token t goes to an expert on host H.
void host_mask(const oracle_problem* p, const Placement& pl, const int32_t* ids,
               std::vector<uint8_t>* mask) {
    mask->assign((size_t)p->T * pl.H, 0);
    for (int t = 0; t < p->T; ++t)
        for (int j = 0; j < p->k; ++j) {
            const int r = pl.rank_of_expert[ids[(size_t)t * p->k + j]];
            (*mask)[(size_t)t * pl.H + r / pl.P] = 1;
        }
}

}  // namespace

extern "C" {

uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    const uint32_t exp_all_ones = 0x7f800000u;
    if ((u & 0x7fffffffu) > exp_all_ones) {
        // NaN: keep sign and top mantissa bits, force a quiet NaN.
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    // Keep the upper 16 bits; the dropped lower 16 bits decide the rounding:
    // above one half ulp round up, below round down, exactly one half round to
    // the even upper value.  A carry out of the mantissa correctly bumps the
    // exponent (and reaches infinity from the largest finite values).
    uint32_t upper = u >> 16;
    const uint32_t dropped = u & 0xffffu;
    const uint32_t half = 0x8000u;
    if (dropped > half || (dropped == half && (upper & 1u))) upper += 1;
    return (uint16_t)upper;
}

float oracle_bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

int oracle_layout(const oracle_problem* p, const int32_t* ids,
                  int32_t* expert_count, int32_t* expert_offset,
                  int32_t* rank_count, int32_t* rank_offset,
                  int32_t* host_count, int32_t* host_offset,
                  uint8_t* mask, int32_t* pos, int32_t* recv_src) {
    Placement pl;
    if (!make_placement(p, &pl)) return ORACLE_ERR_INVALID;
    if (!ids_valid(p, ids)) return ORACLE_ERR_BAD_IDS;
    const int64_t S = (int64_t)p->T * p->k;

    // 1. counts by expert and by rank.
    for (int e = 0; e < p->E; ++e) expert_count[e] = 0;
    for (int r = 0; r < p->R; ++r) rank_count[r] = 0;
    for (int64_t s = 0; s < S; ++s) {
        expert_count[ids[s]] += 1;
        rank_count[pl.rank_of_expert[ids[s]]] += 1;
    }

    // 2. receive order: stable sort of slot indices by (rank(e), e).
    std::vector<int64_t> order(S);
    for (int64_t s = 0; s < S; ++s) order[s] = s;
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
        const int ea = ids[a], eb = ids[b];
        const int ra = pl.rank_of_expert[ea], rb = pl.rank_of_expert[eb];
        if (ra != rb) return ra < rb;
        return ea < eb;
    });
    for (int64_t i = 0; i < S; ++i) {
        pos[order[i]] = (int32_t)i;
        recv_src[i] = (int32_t)order[i];
    }

    // 3. offsets: rank offsets are the exclusive scan over ranks; an expert's
    //    offset is where its segment starts in the receive order.
    rank_offset[0] = 0;
    for (int r = 0; r < p->R; ++r) rank_offset[r + 1] = rank_offset[r] + rank_count[r];
    for (int e = 0; e < p->E; ++e) {
        int32_t start = rank_offset[pl.rank_of_expert[e]];
        for (int e2 = 0; e2 < e; ++e2)
            if (pl.rank_of_expert[e2] == pl.rank_of_expert[e]) start += expert_count[e2];
        expert_offset[e] = start;
    }
    expert_offset[p->E] = (int32_t)S;

    // 4. per-(token, host) mask and de-duplicated per-host token counts.
    std::vector<uint8_t> m;
    host_mask(p, pl, ids, &m);
    std::memcpy(mask, m.data(), m.size());
    for (int H = 0; H < pl.H; ++H) {
        host_count[H] = 0;
        for (int t = 0; t < p->T; ++t) host_count[H] += m[(size_t)t * pl.H + H];
    }
    host_offset[0] = 0;
    for (int H = 0; H < pl.H; ++H) host_offset[H + 1] = host_offset[H] + host_count[H];
    return ORACLE_OK;
}

int oracle_stats(const oracle_problem* p, const int32_t* ids,
                 int64_t* glob, double* ratio, int64_t* src, int64_t* dst) {
    Placement pl;
    if (!make_placement(p, &pl)) return ORACLE_ERR_INVALID;
    std::vector<int32_t> src_of;
    if (!make_sources(p, &src_of)) return ORACLE_ERR_INVALID;
    if (!ids_valid(p, ids)) return ORACLE_ERR_BAD_IDS;
    const int T = p->T, k = p->k, R = p->R, Rs = p->R_src, P = pl.P, H = pl.H;
    const int64_t S = (int64_t)T * k;

    // Row bytes: payload h*elem_bytes, plus one fp32 per scale group for fp8.
    int64_t rho = (int64_t)p->h * p->elem_bytes;
    if (p->elem_bytes == 1) rho += 4LL * (p->h / p->scale_group);

    std::vector<int64_t> ecount(p->E, 0), rslots(R, 0), rtokens(R, 0);
    for (int64_t s = 0; s < S; ++s) {
        ecount[ids[s]] += 1;
        rslots[pl.rank_of_expert[ids[s]]] += 1;
    }
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r) {
            bool hit = false;
            for (int j = 0; j < k; ++j) hit = hit || pl.rank_of_expert[ids[(size_t)t * k + j]] == r;
            if (hit) rtokens[r] += 1;
        }

    std::vector<uint8_t> m;
    host_mask(p, pl, ids, &m);

    // Source side ("Balancing and Beyond" section 3.2): Mode 0 sends every
    // copy that leaves the GPU, Mode 1 one network copy per remote expert,
    // Mode 2 one network copy per remote host holding any of the experts.
    std::vector<int64_t> stok(Rs, 0), mode0(Rs, 0), mode1(Rs, 0), mode2(Rs, 0);
    // Destination side ("Profiling when rank unbalance"): slots a rank
    // receives from itself, from other ranks of its host, from other hosts;
    // and Mode 2 network copies landing on the same-index relay GPU.
    std::vector<int64_t> rself(R, 0), rlocal(R, 0), rremote(R, 0), rrelay(R, 0);
    for (int t = 0; t < T; ++t) {
        const int rs = src_of[t];
        stok[rs] += 1;
        for (int j = 0; j < k; ++j) {
            const int rd = pl.rank_of_expert[ids[(size_t)t * k + j]];
            if (rd != rs) mode0[rs] += 1;
            if (rd / P != rs / P) mode1[rs] += 1;
            if (rd == rs) rself[rd] += 1;
            else if (rd / P == rs / P) rlocal[rd] += 1;
            else rremote[rd] += 1;
        }
        for (int hh = 0; hh < H; ++hh) {
            if (hh == rs / P || !m[(size_t)t * H + hh]) continue;
            mode2[rs] += 1;
            rrelay[hh * P + rs % P] += 1;
        }
    }

    for (int i = 0; i < ORACLE_STATS_GLOBAL_WORDS; ++i) glob[i] = 0;
    glob[ORACLE_G_T] = T;
    glob[ORACLE_G_SLOTS] = S;
    glob[ORACLE_G_ROW_BYTES] = rho;
    int64_t mx = -1, mn = -1, amx = 0;
    for (int e = 0; e < p->E; ++e) {
        if (ecount[e] > mx) { mx = ecount[e]; amx = e; }
        if (mn < 0 || ecount[e] < mn) mn = ecount[e];
    }
    glob[ORACLE_G_MAX_EXPERT] = mx;
    glob[ORACLE_G_ARGMAX_EXPERT] = amx;
    glob[ORACLE_G_MIN_EXPERT] = mn;
    // Imbalance ratio: busiest expert over the layer mean T*k/E
    // ("Balancing and Beyond" section 2).
    ratio[0] = S > 0 ? (double)mx / ((double)S / (double)p->E) : 0.0;
    int64_t mrs = 0, mrt = 0;
    for (int r = 0; r < R; ++r) { mrs = std::max(mrs, rslots[r]); mrt = std::max(mrt, rtokens[r]); }
    glob[ORACLE_G_MAX_RANK_SLOTS] = mrs;
    glob[ORACLE_G_MAX_RANK_TOKENS] = mrt;
    ratio[1] = S > 0 ? (double)mrs / ((double)S / (double)R) : 0.0;

    for (int r = 0; r < Rs; ++r) {
        const int64_t copies = stok[r] * k;
        src[0 * Rs + r] = stok[r];
        src[1 * Rs + r] = copies;
        src[2 * Rs + r] = mode0[r];
        src[3 * Rs + r] = mode1[r];
        src[4 * Rs + r] = mode2[r];
        // "tokens x k x h x 2 B" leave a GPU per layer and direction
        // ("Balancing and Beyond" section 1).
        src[5 * Rs + r] = stok[r] * k * (int64_t)p->h * 2;
        src[6 * Rs + r] = mode0[r] * rho;
        src[7 * Rs + r] = mode1[r] * rho;
        src[8 * Rs + r] = mode2[r] * rho;
        glob[ORACLE_G_SUM_MODE0] += mode0[r];
        glob[ORACLE_G_SUM_MODE1] += mode1[r];
        glob[ORACLE_G_SUM_MODE2] += mode2[r];
        glob[ORACLE_G_MAX_SRC_MODE1] = std::max(glob[ORACLE_G_MAX_SRC_MODE1], mode1[r]);
        glob[ORACLE_G_MAX_SRC_MODE2] = std::max(glob[ORACLE_G_MAX_SRC_MODE2], mode2[r]);
        glob[ORACLE_G_SUM_NAIVE_BYTES] += src[5 * Rs + r];
        glob[ORACLE_G_SUM_MODE0_BYTES] += src[6 * Rs + r];
        glob[ORACLE_G_SUM_MODE1_BYTES] += src[7 * Rs + r];
        glob[ORACLE_G_SUM_MODE2_BYTES] += src[8 * Rs + r];
    }
    for (int r = 0; r < R; ++r) {
        dst[0 * R + r] = rslots[r];
        dst[1 * R + r] = rtokens[r];
        dst[2 * R + r] = rself[r];
        dst[3 * R + r] = rlocal[r];
        dst[4 * R + r] = rremote[r];
        dst[5 * R + r] = rrelay[r];
        glob[ORACLE_G_MAX_RECV_REMOTE] = std::max(glob[ORACLE_G_MAX_RECV_REMOTE], rremote[r]);
        glob[ORACLE_G_MAX_RECV_RELAY] = std::max(glob[ORACLE_G_MAX_RECV_RELAY], rrelay[r]);
    }
    return ORACLE_OK;
}

void oracle_dispatch(const oracle_problem* p, const int32_t* pos,
                     const uint8_t* x, const float* x_scales,
                     uint8_t* recv, float* recv_scales) {
    const size_t row = (size_t)p->h * p->elem_bytes;
    const size_t groups = p->elem_bytes == 1 ? (size_t)(p->h / p->scale_group) : 0;
    for (int t = 0; t < p->T; ++t)
        for (int j = 0; j < p->k; ++j) {
            const size_t dst_row = (size_t)pos[(size_t)t * p->k + j];
            std::memcpy(recv + dst_row * row, x + (size_t)t * row, row);
            if (groups && x_scales && recv_scales)
                std::memcpy(recv_scales + dst_row * groups, x_scales + (size_t)t * groups,
                            groups * sizeof(float));
        }
}

int oracle_relay_layout(const oracle_problem* p, const int32_t* ids, int32_t* relay_pos) {
    Placement pl;
    if (!make_placement(p, &pl)) return ORACLE_ERR_INVALID;
    if (!ids_valid(p, ids)) return ORACLE_ERR_BAD_IDS;
    std::vector<uint8_t> m;
    host_mask(p, pl, ids, &m);
    // Relay segments in host order; inside a segment, ascending token order.
    std::vector<int32_t> start(pl.H + 1, 0);
    for (int hh = 0; hh < pl.H; ++hh) {
        int32_t c = 0;
        for (int t = 0; t < p->T; ++t) c += m[(size_t)t * pl.H + hh];
        start[hh + 1] = start[hh] + c;
    }
    for (int hh = 0; hh < pl.H; ++hh) {
        int32_t next = start[hh];
        for (int t = 0; t < p->T; ++t)
            relay_pos[(size_t)t * pl.H + hh] = m[(size_t)t * pl.H + hh] ? next++ : -1;
    }
    return ORACLE_OK;
}

void oracle_relay_dispatch(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                           const int32_t* relay_pos, const uint8_t* x, const float* x_scales,
                           uint8_t* relay, float* relay_scales, uint8_t* recv, float* recv_scales) {
    Placement pl;
    make_placement(p, &pl);
    const size_t row = (size_t)p->h * p->elem_bytes;
    const size_t groups = p->elem_bytes == 1 ? (size_t)(p->h / p->scale_group) : 0;
    // hop 1: one copy per (token, host)
    for (int t = 0; t < p->T; ++t)
        for (int hh = 0; hh < pl.H; ++hh) {
            const int32_t r = relay_pos[(size_t)t * pl.H + hh];
            if (r < 0) continue;
            std::memcpy(relay + (size_t)r * row, x + (size_t)t * row, row);
            if (groups) std::memcpy(relay_scales + (size_t)r * groups, x_scales + (size_t)t * groups, groups * 4);
        }
    // hop 2: fan-out on the host, from the relay row
    for (int t = 0; t < p->T; ++t)
        for (int j = 0; j < p->k; ++j) {
            const int hh = pl.rank_of_expert[ids[(size_t)t * p->k + j]] / pl.P;
            const int32_t r = relay_pos[(size_t)t * pl.H + hh];
            const size_t dst = (size_t)pos[(size_t)t * p->k + j];
            std::memcpy(recv + dst * row, relay + (size_t)r * row, row);
            if (groups) std::memcpy(recv_scales + dst * groups, relay_scales + (size_t)r * groups, groups * 4);
        }
}

void oracle_relay_combine(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                          const int32_t* relay_pos, const uint16_t* y, const float* w,
                          uint16_t* partial, uint16_t* out) {
    Placement pl;
    make_placement(p, &pl);
    const size_t h = (size_t)p->h;
    // hop 1: per (token, host) partial sums, rounded to bf16 as they travel
    for (int t = 0; t < p->T; ++t)
        for (int hh = 0; hh < pl.H; ++hh) {
            const int32_t r = relay_pos[(size_t)t * pl.H + hh];
            if (r < 0) continue;
            for (size_t c = 0; c < h; ++c) {
                float acc = 0.0f;
                for (int j = 0; j < p->k; ++j) {
                    if (pl.rank_of_expert[ids[(size_t)t * p->k + j]] / pl.P != hh) continue;
                    const size_t src = (size_t)pos[(size_t)t * p->k + j];
                    acc = std::fma(w[(size_t)t * p->k + j], oracle_bf16_to_f32(y[src * h + c]), acc);
                }
                partial[(size_t)r * h + c] = oracle_f32_to_bf16_rne(acc);
            }
        }
    // hop 2: the token's partials summed in ascending host order
    for (int t = 0; t < p->T; ++t)
        for (size_t c = 0; c < h; ++c) {
            float acc = 0.0f;
            for (int hh = 0; hh < pl.H; ++hh) {
                const int32_t r = relay_pos[(size_t)t * pl.H + hh];
                if (r >= 0) acc = acc + oracle_bf16_to_f32(partial[(size_t)r * h + c]);
            }
            out[(size_t)t * h + c] = oracle_f32_to_bf16_rne(acc);
        }
}

int oracle_expert_groups(const oracle_problem* p, int G, int32_t* group) {
    Placement pl;
    if (!make_placement(p, &pl) || G < 1) return ORACLE_ERR_INVALID;
    std::vector<int32_t> n(pl.R, 0), li(pl.E, 0);
    for (int e = 0; e < pl.E; ++e) li[e] = n[pl.rank_of_expert[e]]++;  // ascending e inside a rank
    for (int e = 0; e < pl.E; ++e)
        group[e] = (int32_t)(((int64_t)li[e] * G) / n[pl.rank_of_expert[e]]);
    return ORACLE_OK;
}

void oracle_dispatch_group(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                           const int32_t* group, int g, const uint8_t* x, const float* x_scales,
                           uint8_t* recv, float* recv_scales) {
    const size_t row = (size_t)p->h * p->elem_bytes;
    const size_t groups = p->elem_bytes == 1 ? (size_t)(p->h / p->scale_group) : 0;
    for (int t = 0; t < p->T; ++t)
        for (int j = 0; j < p->k; ++j) {
            const size_t s = (size_t)t * p->k + j;
            if (group[ids[s]] != g) continue;
            const size_t dst = (size_t)pos[s];
            std::memcpy(recv + dst * row, x + (size_t)t * row, row);
            if (groups) std::memcpy(recv_scales + dst * groups, x_scales + (size_t)t * groups, groups * 4);
        }
}

void oracle_combine_group(const oracle_problem* p, const int32_t* ids, const int32_t* pos,
                          const int32_t* group, int g, int G, const uint16_t* y, const float* w,
                          float* acc, uint16_t* out) {
    const size_t h = (size_t)p->h;
    for (int t = 0; t < p->T; ++t)
        for (size_t c = 0; c < h; ++c) {
            float a = g == 0 ? 0.0f : acc[(size_t)t * h + c];
            for (int j = 0; j < p->k; ++j) {
                const size_t s = (size_t)t * p->k + j;
                if (group[ids[s]] != g) continue;
                a = std::fma(w[s], oracle_bf16_to_f32(y[(size_t)pos[s] * h + c]), a);
            }
            if (g == G - 1)
                out[(size_t)t * h + c] = oracle_f32_to_bf16_rne(a);
            else
                acc[(size_t)t * h + c] = a;
        }
}

int oracle_swap_plan(const oracle_problem* p, const int32_t* expert_count, int32_t tau,
                     int32_t* new_expert_to_rank, int32_t* swaps) {
    Placement pl;
    if (!make_placement(p, &pl)) return ORACLE_ERR_INVALID;
    const int P = pl.P, H = pl.H, pairs = P / 2;
    std::vector<int64_t> load(p->R, 0);
    for (int e = 0; e < p->E; ++e) load[pl.rank_of_expert[e]] += expert_count[e];
    for (int e = 0; e < p->E; ++e) new_expert_to_rank[e] = pl.rank_of_expert[e];
    const int64_t need = std::max<int64_t>(tau, 1);
    for (int hh = 0; hh < H; ++hh) {
        // Ranks of the host, heaviest first (ties by rank index).
        std::vector<int> ranks(P);
        for (int i = 0; i < P; ++i) ranks[i] = hh * P + i;
        std::stable_sort(ranks.begin(), ranks.end(), [&](int x, int y) { return load[x] > load[y]; });
        for (int i = 0; i < pairs; ++i) {
            const int a = ranks[i], b = ranks[P - 1 - i];
            const int64_t old_max = std::max(load[a], load[b]);
            int64_t best = -1;
            int bx = -1, by = -1;
            for (int x = 0; x < p->E; ++x) {
                if (pl.rank_of_expert[x] != a) continue;
                for (int y = 0; y < p->E; ++y) {
                    if (pl.rank_of_expert[y] != b) continue;
                    const int64_t la = load[a] - expert_count[x] + expert_count[y];
                    const int64_t lb = load[b] - expert_count[y] + expert_count[x];
                    const int64_t m = std::max(la, lb);
                    if (best < 0 || m < best) { best = m; bx = x; by = y; }
                }
            }
            int32_t* rec = swaps + ((size_t)hh * pairs + i) * 6;
            rec[0] = a; rec[1] = b; rec[2] = bx; rec[3] = by;
            rec[4] = (int32_t)old_max;
            rec[5] = (int32_t)(best < 0 ? old_max : best);
            if (bx >= 0 && old_max - best >= need) {
                new_expert_to_rank[bx] = b;
                new_expert_to_rank[by] = a;
            }
        }
    }
    return ORACLE_OK;
}

float oracle_e4m3_to_f32(uint8_t c) {
    const int sign = (c >> 7) & 1;
    const int exp = (c >> 3) & 0xF;
    const int man = c & 0x7;
    if (exp == 0xF && man == 0x7) return std::nanf("");
    float mag;
    if (exp == 0) mag = std::ldexp((float)man / 8.0f, 1 - 7);           // subnormal: 0.m x 2^-6
    else mag = std::ldexp(1.0f + (float)man / 8.0f, exp - 7);            // normal: 1.m x 2^(e-7)
    return sign ? -mag : mag;
}

uint8_t oracle_f32_to_e4m3_sat(float f) {
    if (std::isnan(f)) return 0x7F;
    const uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
    const double a = std::fabs((double)f);
    // Every non-negative finite code in ascending order of value: codes 0x00
    // .. 0x7E (0x7F is NaN).  Pick the nearest; on an exact tie the even code
    // (lowest mantissa bit 0); beyond the largest (448) saturate.
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = a;  // distance to code 0 (value 0)
    for (int c = 1; c <= 0x7E; ++c) {
        const double v = (double)oracle_e4m3_to_f32((uint8_t)c);
        const double d = std::fabs(v - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

void oracle_quantize_dispatch(const oracle_problem* p, const int32_t* pos, const uint16_t* x_bf16,
                              uint8_t* recv_codes, float* recv_scales) {
    const size_t h = (size_t)p->h, g = (size_t)p->scale_group, G = h / g;
    std::vector<uint8_t> codes(h);
    std::vector<float> scales(G);
    for (int t = 0; t < p->T; ++t) {
        const uint16_t* row = x_bf16 + (size_t)t * h;
        for (size_t grp = 0; grp < G; ++grp) {
            float amax = 0.0f;
            for (size_t c = grp * g; c < (grp + 1) * g; ++c)
                amax = std::max(amax, std::fabs(oracle_bf16_to_f32(row[c])));
            const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[grp] = scale;
            for (size_t c = grp * g; c < (grp + 1) * g; ++c)
                codes[c] = oracle_f32_to_e4m3_sat(oracle_bf16_to_f32(row[c]) / scale);
        }
        for (int j = 0; j < p->k; ++j) {
            const size_t dst = (size_t)pos[(size_t)t * p->k + j];
            std::memcpy(recv_codes + dst * h, codes.data(), h);
            std::memcpy(recv_scales + dst * G, scales.data(), G * sizeof(float));
        }
    }
}

void oracle_combine(const oracle_problem* p, const int32_t* pos,
                    const uint16_t* y, const float* w, uint16_t* out) {
    const size_t h = (size_t)p->h;
    for (int t = 0; t < p->T; ++t)
        for (size_t c = 0; c < h; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < p->k; ++j) {
                const size_t src_row = (size_t)pos[(size_t)t * p->k + j];
                acc = std::fma(w[(size_t)t * p->k + j], oracle_bf16_to_f32(y[src_row * h + c]), acc);
            }
            out[(size_t)t * h + c] = oracle_f32_to_bf16_rne(acc);
        }
}

}  // extern "C"
