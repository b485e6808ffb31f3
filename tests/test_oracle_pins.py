"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

None of these compares the oracle with itself.  Each pin is one of: a closed
form the pages print, a worked example the pages print, a byte count the pages
print, a brute-force enumeration of a definition on tiny inputs, or a library
routine that a special case reduces to.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import moe_workloads as mw


def golden(name):
    """A worked example the pages print (tests/golden/page_values.json)."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_values.json")
    return json.load(open(path))[name]


def _prob(oracle, T, E, R, P, k, h=8, R_src=1, elem_bytes=2, e2r=None, src_off=None):
    return oracle.make_problem(T, h, k, E, R, P, R_src, elem_bytes, 128, e2r, src_off)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rne_matches_library_conversion(oracle_mod):
    """bf16 round-to-nearest-even: the oracle's bit rule equals torch's conversion."""
    import torch
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(4000).astype(np.float32),
            (rng.standard_normal(2000) * 1e30).astype(np.float32),
            (rng.standard_normal(2000) * 1e-38).astype(np.float32)]  # subnormals
    # exact ties: upper bits even/odd with dropped half = 0x8000
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x7F7F8000, 0x00018000, 0x3F80FFFF,
                     0x3F807FFF, 0x7F7FFFFF, 0x00000000, 0x80000000, 0x7F800000, 0xFF800000],
                    dtype=np.uint32).view(np.float32)
    v = np.concatenate(vals + [ties])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.f32_to_bf16(v)
    assert np.array_equal(got, want)
    back = oracle_mod.bf16_to_f32(got)
    assert np.array_equal(back.view(np.uint32), got.astype(np.uint32) << 16)


# ------------------------------------------------------- layout by brute force

def _brute_layout(ids, rank_of, H, P):
    """pos by counting (not sorting): slots with a smaller (rank, expert) key,
    plus earlier tokens of the same expert."""
    T, k = ids.shape
    key = lambda e: (rank_of[e], e)  # noqa: E731
    pos = np.zeros((T, k), np.int64)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            n = 0
            for t2 in range(T):
                for j2 in range(k):
                    e2 = ids[t2, j2]
                    if key(e2) < key(e) or (e2 == e and t2 < t):
                        n += 1
            pos[t, j] = n
    mask = np.zeros((T, H), np.uint8)
    for t in range(T):
        for j in range(k):
            mask[t, rank_of[ids[t, j]] // P] = 1
    return pos, mask


@pytest.mark.parametrize("e2r", [None, [1, 0, 1, 0], [0, 0, 1, 1], [1, 1, 1, 0]])
def test_layout_exhaustive_tiny(oracle_mod, e2r):
    """Every id assignment of 3 tokens x 2 distinct experts out of 4, two ranks
    on two hosts, against the counting definition of the receive order."""
    E, k, T, R, P = 4, 2, 3, 2, 1
    rank_of = [e // 2 for e in range(E)] if e2r is None else e2r
    pairs = [p for p in itertools.permutations(range(E), k)]
    prob, keep = _prob(oracle_mod, T, E, R, P, k, e2r=e2r)
    for combo in itertools.product(pairs, repeat=T):
        ids = np.array(combo, np.int32)
        lay = oracle_mod.layout(prob, ids)
        pos, mask = _brute_layout(ids, rank_of, R // P, P)
        assert np.array_equal(lay["pos"], pos)
        assert np.array_equal(lay["host_mask"], mask)
        cnt = np.bincount(ids.ravel(), minlength=E)
        assert np.array_equal(lay["expert_count"], cnt)
        for e in range(E):
            assert lay["expert_offset"][e] == sum(cnt[e2] for e2 in range(E)
                                                  if (rank_of[e2], e2) < (rank_of[e], e))


@pytest.mark.parametrize("name", ["tiny", "decode-EP32-r8", "decode-EP32-alt", "prefill"])
def test_layout_invariants(oracle_mod, name):
    w = mw.WORKLOADS[name]
    if w.T > 1024:
        w = mw.scaled(w, T=1024, R_src=min(w.R_src, 8))
    ids = mw.gen_ids(w, step=3 % w.steps)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, R_src=w.R_src)
    lay = oracle_mod.layout(prob, ids)
    S = w.T * w.k
    rank_of = np.arange(w.E) // (w.E // w.R)
    assert lay["expert_count"].sum() == S
    assert np.array_equal(lay["rank_count"], np.bincount(rank_of, weights=lay["expert_count"],
                                                         minlength=w.R).astype(np.int64))
    assert np.array_equal(lay["rank_offset"], np.concatenate([[0], np.cumsum(lay["rank_count"])]))
    pos = lay["pos"].ravel()
    assert np.array_equal(np.sort(pos), np.arange(S))            # bijection onto [0, T*k)
    assert np.array_equal(lay["recv_src"][pos], np.arange(S))    # inverse map
    # library routine: numpy's lexsort by (rank, expert), ties by slot index
    flat = ids.ravel()
    order = np.lexsort((np.arange(S), flat, rank_of[flat]))
    assert np.array_equal(lay["recv_src"], order)
    for e in range(w.E):  # expert segments: contiguous, ascending token order
        seg = lay["recv_src"][lay["expert_offset"][e]:lay["expert_offset"][e] + lay["expert_count"][e]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // w.k) > 0)
    assert np.array_equal(lay["host_count"], lay["host_mask"].sum(axis=0))
    assert np.array_equal(lay["host_offset"], np.concatenate([[0], np.cumsum(lay["host_count"])]))


def test_oracle_rejects_bad_ids(oracle_mod):
    prob, keep = _prob(oracle_mod, 2, 4, 2, 1, 2)
    with pytest.raises(oracle_mod.OracleError) as ei:
        oracle_mod.layout(prob, np.array([[0, 0], [1, 2]], np.int32))
    assert ei.value.code == oracle_mod.ERR_BAD_IDS
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.layout(prob, np.array([[0, 4], [1, 2]], np.int32))
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.stats(prob, np.array([[-1, 1], [1, 2]], np.int32))


# ------------------------------------------- copy counts: closed forms (c0, c1, c2)

def _c2(E, k, H):
    """Mode 2 copies per token ("Balancing and Beyond", section 3.2)."""
    return Fraction(H - 1) * (1 - Fraction(math.comb(E - E // H, k), math.comb(E, k)))


@pytest.mark.parametrize("E,k,R,P", [(16, 2, 4, 2), (12, 3, 6, 2), (8, 2, 4, 1), (16, 3, 8, 2)])
def test_copy_counts_exact_over_all_expert_sets(oracle_mod, E, k, R, P):
    """Averaged over all C(E, k) expert sets, the per-token copy counts are
    exactly c0 = k(1 - 1/EP), c1 = k(H-1)/H and c2 = (H-1)[1 - C(E-E/H, k)/C(E, k)]."""
    H = R // P
    subsets = np.array(list(itertools.combinations(range(E), k)), np.int32)
    T = len(subsets)
    prob, keep = _prob(oracle_mod, T, E, R, P, k, R_src=1)  # every token on rank 0
    st = oracle_mod.stats(prob, subsets)
    assert Fraction(int(st["src_mode0"][0]), T) == Fraction(k) * (1 - Fraction(1, R))
    assert Fraction(int(st["src_mode1"][0]), T) == Fraction(k * (H - 1), H)
    assert Fraction(int(st["src_mode2"][0]), T) == _c2(E, k, H)


def test_copy_counts_tiny_value(oracle_mod):
    """E=16, k=2, H=2: c1 = 1 and c2 = 23/30 exactly."""
    assert _c2(16, 2, 2) == Fraction(23, 30)
    subsets = np.array(list(itertools.combinations(range(16), 2)), np.int32)
    prob, keep = _prob(oracle_mod, len(subsets), 16, 4, 2, 2, R_src=1)
    st = oracle_mod.stats(prob, subsets)
    assert (st["src_mode1"][0], st["src_mode2"][0]) == (120, 92)


def test_copy_counts_deepseek_shape(oracle_mod):
    """E=256, k=8, EP32 on four hosts: c1 = 6, c2 ~ 2.7, 55 % fewer network
    copies ("Balancing and Beyond", section 3.2); uniform sample, 4 sigma."""
    g = golden("dedup_deepseek")
    E, k, R, H = g["experts"], g["topk"], g["ranks"], g["hosts"]
    w = mw.Workload("u", T=20000, h=8, k=k, E=E, R=R, P=R // H, R_src=1, seed=11)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, R_src=1)
    st = oracle_mod.stats(prob, ids)
    c1 = st["src_mode1"][0] / w.T
    c2 = st["src_mode2"][0] / w.T
    c2_exact = float(_c2(E, k, H))
    assert abs(c2_exact - 2.7107) < 1e-4 and round(c2_exact, 1) == g["c2_approx"]
    # per-token variances are at most k p (1 - p) = 1.5 (c1) and 0.75 (c2)
    assert abs(c1 - g["c1"]) < 4 * math.sqrt(1.5 / w.T)
    assert abs(c2 - c2_exact) < 4 * math.sqrt(0.75 / w.T)
    assert round(1 - c2_exact / g["c1"], 2) == g["fewer_network_bytes"]


def test_hybridep_rdma_send_bytes(oracle_mod):
    """The HybridEP issue's shape (4096 tokens, h=7168, 16 ranks on 2 hosts, 8
    local experts, top-8) prints rdma_send_bytes 117.11 MB (bf16) and 60.40 MB
    (fp8 with scales): one copy per (token, host) over all hosts.  Uniform
    routing; tolerance 3.5 sampling sigmas (0.25 MB)."""
    g = golden("hybridep_rdma_send_bytes")
    w = mw.WORKLOADS["prefill"]
    assert (w.T, w.h, w.R, w.R // w.P, w.E // w.R, w.k) == (g["tokens"], g["hidden"], g["ranks"], g["hosts"],
                                                           g["local_experts"], g["topk"])
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=1)
    lay = oracle_mod.layout(prob, ids)
    st_bf16 = oracle_mod.stats(prob, ids)
    probf, keepf = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=1, elem_bytes=1)
    st_fp8 = oracle_mod.stats(probf, ids)
    assert st_bf16["row_bytes"] == 14336 and st_fp8["row_bytes"] == 7168 + 4 * 56
    copies = int(lay["host_count"].sum())
    assert abs(copies * st_bf16["row_bytes"] - g["bf16_MB"] * 1e6) < 0.25e6
    assert abs(copies * st_fp8["row_bytes"] - g["fp8_MB"] * 1e6) < 0.13e6


# --------------------------------------------- "Profiling when rank unbalance"

def _p1_case(oracle_mod, per_rank):
    """16 ranks on 2 hosts, one expert per rank, k=1; a source rank sends its
    i-th token to rank i mod 16."""
    R, P = 16, 8
    src_off = np.concatenate([[0], np.cumsum(per_rank)]).astype(np.int32)
    ids = np.concatenate([np.arange(n) % R for n in per_rank]).astype(np.int32)[:, None]
    prob, keep = _prob(oracle_mod, int(src_off[-1]), R, R, P, 1, R_src=R, src_off=src_off)
    return oracle_mod.stats(prob, ids)


def test_p1_unbalanced_receive_counts(oracle_mod):
    """Host-0 ranks hold 384 tokens, host-1 ranks 64: a host-1 rank receives
    (384/16)*8 = 192 from host 0 and (64/16)*7 = 28 from its own host, 220 in
    all; each host-0 GPU sends 192 tokens over the network."""
    g = golden("unbalanced_batch")
    st = _p1_case(oracle_mod, [g["tokens_per_rank_host0"]] * 8 + [g["tokens_per_rank_host1"]] * 8)
    for r in range(8, 16):
        assert st["recv_remote"][r] == g["host1_rank_recv_from_host0"]
        assert st["recv_local"][r] == g["host1_rank_recv_from_own_host"]
        assert st["recv_remote"][r] + st["recv_local"][r] == g["host1_rank_recv_total"]
    for r in range(8):
        assert st["src_mode1"][r] == g["host0_gpu_sends_unbalanced"]


def test_p1_balanced_receive_counts(oracle_mod):
    """224 tokens per rank: (224/16)*15 = 210 received from other ranks, 112 of
    them over the network; each GPU sends 112 over the network."""
    g = golden("unbalanced_batch")
    st = _p1_case(oracle_mod, [g["balanced_tokens_per_rank"]] * 16)
    for r in range(16):
        assert st["recv_remote"][r] + st["recv_local"][r] == g["balanced_recv_from_other_ranks"]
        assert st["recv_remote"][r] == g["balanced_recv_over_network"]
        assert st["src_mode1"][r] == g["gpu_sends_balanced"]


# ------------------------------------------------------------- imbalance ratio

def test_imbalance_ratio_special_cases(oracle_mod):
    E, k, T = 16, 2, 64
    prob, keep = _prob(oracle_mod, T, E, 4, 2, k, R_src=1)
    same = np.tile(np.array([[3, 9]], np.int32), (T, 1))
    assert oracle_mod.stats(prob, same)["imbalance_ratio"] == E / k
    rr = (np.arange(T * k) % E).astype(np.int32).reshape(T, k)
    st = oracle_mod.stats(prob, rr)
    assert st["imbalance_ratio"] == 1.0 and st["rank_imbalance"] == 1.0


def test_bytes_formulas(oracle_mod):
    """tokens x k x h x 2 B per rank and direction, copies x row bytes per mode."""
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=512, R_src=32)
    ids = mw.gen_ids(w)
    for eb in (2, 1):
        prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=w.R_src, elem_bytes=eb)
        st = oracle_mod.stats(prob, ids)
        rho = w.h * 2 if eb == 2 else w.h + 4 * (w.h // 128)
        assert st["row_bytes"] == rho
        assert np.all(st["src_naive_bytes"] == st["src_tokens"] * w.k * w.h * 2)
        assert np.all(st["src_copies"] == st["src_tokens"] * w.k)
        for m in (0, 1, 2):
            assert np.all(st[f"src_mode{m}_bytes"] == st[f"src_mode{m}"] * rho)
        assert np.all(st["src_mode2"] <= st["src_mode1"])
        assert np.all(st["src_mode1"] <= st["src_mode0"])
        assert st["recv_slots"].sum() == w.T * w.k
        assert np.array_equal(st["recv_self"] + st["recv_local"] + st["recv_remote"], st["recv_slots"])
        assert st["recv_relay"].sum() == st["sum_mode2_copies"]


# -------------------------------------------------------- dispatch and combine

def test_dispatch_moves_rows(oracle_mod):
    w = mw.scaled(mw.WORKLOADS["tiny"], T=64)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=w.R_src)
    lay = oracle_mod.layout(prob, ids)
    x = mw.gen_x_bf16(w)
    recv = oracle_mod.dispatch(prob, lay["pos"], x)
    assert np.array_equal(recv[lay["pos"]], np.repeat(x[:, None, :], w.k, axis=1))
    wf = mw.scaled(w, dtype="fp8")
    probf, keepf = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=w.R_src, elem_bytes=1)
    q, sc = mw.gen_x_fp8(wf)
    rq, rs = oracle_mod.dispatch(probf, lay["pos"], q, sc)
    src_tok = lay["recv_src"] // w.k
    assert np.array_equal(rq, q[src_tok]) and np.array_equal(rs, sc[src_tok])


@pytest.mark.parametrize("k", [2, 8])
def test_combine_unit_weights_identity_experts(oracle_mod, k):
    """Permute then unpermute with identity experts and unit weights returns
    k * x exactly (k a power of two)."""
    w = mw.Workload("rt", T=96, h=256, k=k, E=32, R=8, P=4, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    x = mw.gen_x_bf16(w)
    recv = oracle_mod.dispatch(prob, lay["pos"], x)
    out = oracle_mod.combine(prob, lay["pos"], recv, np.ones((w.T, k), np.float32))
    want = mw.bf16_bits_to_f32(x) * np.float32(k)
    # equal as values (an input -0.0 sums to +0.0 from the +0.0 start)
    assert np.array_equal(mw.bf16_bits_to_f32(out), want)
    neg0 = oracle_mod.combine(prob, lay["pos"][:1], np.full((w.slots, w.h), 0x8000, np.uint16),
                              np.ones((1, k), np.float32))
    assert np.all(neg0[0] == 0x0000)


def test_combine_k1_is_a_gather(oracle_mod):
    w = mw.Workload("k1", T=50, h=64, k=1, E=8, R=4, P=2, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, 1, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    y = mw.gen_y_host(w)
    out = oracle_mod.combine(prob, lay["pos"], y, np.ones((w.T, 1), np.float32))
    assert np.array_equal(out, y[lay["pos"][:, 0]])


def test_combine_error_bound_against_fp64(oracle_mod):
    """|out - sum_j w_j y_j| <= 2^-8 |exact| + (1 + 2^-8) k 2^-24 sum_j |w_j y_j|:
    half a bf16 ulp for the final rounding plus the fp32 fma chain."""
    w = mw.Workload("c", T=128, h=512, k=8, E=64, R=8, P=4, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    y = mw.gen_y_host(w)
    g = mw.gen_gates(w)
    out = mw.bf16_bits_to_f32(oracle_mod.combine(prob, lay["pos"], y, g)).astype(np.float64)
    yf = mw.bf16_bits_to_f32(y).astype(np.float64)[lay["pos"]]           # [T, k, h]
    terms = g.astype(np.float64)[:, :, None] * yf
    exact = terms.sum(axis=1)
    bound = 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * w.k * 2.0 ** -24 * np.abs(terms).sum(axis=1)
    assert np.all(np.abs(out - exact) <= bound)


def test_combine_sums_in_ascending_slot_order(oracle_mod):
    """y rows 2^24, 1, -2^24 with unit weights: ascending slot order gives
    (2^24 + 1) - 2^24 = 0 in fp32 (the tie rounds to even), any order that
    adds the two large terms first gives 1."""
    prob, keep = _prob(oracle_mod, 1, 3, 3, 1, 3, h=8)
    pos = np.array([[0, 1, 2]], np.int32)
    y = mw.f32_to_bf16_bits(np.array([[2.0 ** 24] * 8, [1.0] * 8, [-(2.0 ** 24)] * 8], np.float32))
    out = oracle_mod.combine(prob, pos, y, np.ones((1, 3), np.float32))
    assert np.all(out == 0)
    out_rev = oracle_mod.combine(prob, np.array([[0, 2, 1]], np.int32), y, np.ones((1, 3), np.float32))
    assert np.all(mw.bf16_bits_to_f32(out_rev) == 1.0)


# ------------------------------------------------------- fp8 e4m3 quantisation

def _torch_e4m3_values():
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_matches_library(oracle_mod):
    """All 256 e4m3 codes decode as the library's float8_e4m3fn does (0x7F and
    0xFF are NaN; 0x7E is 448)."""
    want = _torch_e4m3_values()
    got = oracle_mod.e4m3_to_f32(np.arange(256))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0


def test_e4m3_encode_round_trip_ties_and_saturation(oracle_mod):
    vals = _torch_e4m3_values()
    finite = [c for c in range(256) if not np.isnan(vals[c])]
    enc = oracle_mod.f32_to_e4m3(vals[finite])
    # -0.0 encodes to 0x80, +0.0 to 0x00: every finite code round-trips
    assert np.array_equal(enc, np.array(finite, np.uint8))
    # ties between neighbours go to the even code; compare with the library
    import torch
    pos = np.sort(vals[[c for c in range(0x7F) if not np.isnan(vals[c])]])
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    got = oracle_mod.f32_to_e4m3(np.concatenate([mids, -mids]))
    want = torch.from_numpy(np.concatenate([mids, -mids])).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    assert np.all(got[: len(mids)] % 2 == 0)
    # beyond the largest finite value: saturate to +-448
    big = np.array([448.0001, 464.0, 480.0, 1e6, 3.4e38], np.float32)
    assert np.all(oracle_mod.f32_to_e4m3(big) == 0x7E)
    assert np.all(oracle_mod.f32_to_e4m3(-big) == 0xFE)


def test_e4m3_encode_matches_library_rne(oracle_mod):
    import torch
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(3000) * 2.0 ** -7,
                        rng.standard_normal(2000)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.f32_to_e4m3(v), want)


def test_quantize_dispatch_bounds_and_rows(oracle_mod):
    """Per 128-column group: the element of largest magnitude maps to +-448;
    every element dequantises within half an e4m3 ulp (relative 2^-4, or
    2^-10 x scale in the subnormal range); each receive row holds its token's
    quantised row."""
    w = mw.Workload("q", T=48, h=512, k=4, E=16, R=4, P=2, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, elem_bytes=1)
    lay = oracle_mod.layout(prob, ids)
    x = mw.gen_x_bf16(w)
    codes, scales = oracle_mod.quantize_dispatch(prob, lay["pos"], x)
    src = lay["recv_src"] // w.k
    xf = mw.bf16_bits_to_f32(x).reshape(w.T, -1, 128)
    amax = np.abs(xf).max(axis=2)
    assert np.array_equal(scales[lay["pos"][:, 0]], (amax / np.float32(448.0)).astype(np.float32))
    dq = oracle_mod.e4m3_to_f32(codes[lay["pos"][:, 0]]).reshape(w.T, -1, 128)
    scale = scales[lay["pos"][:, 0]][:, :, None]
    err = np.abs(dq.astype(np.float64) * scale - xf)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * scale) * (1 + 1e-6))
    top = np.abs(xf).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(dq, top[:, :, None], axis=2)) == 448.0)
    assert np.array_equal(codes, codes[lay["pos"][:, 0]][src])
    assert np.array_equal(scales, scales[lay["pos"][:, 0]][src])


# ------------------------------------------------ per-step intra-host expert swap

def test_swap_plan_worked_example(oracle_mod):
    """"Balancing and Beyond", Figure 2(b): G0 holds e0 (60 tokens) and 100
    more, G1 holds e1 (30) and 70 more; swapping e0 and e1 turns 160 / 100 into
    130 / 130.  The swap is taken when tau <= 30 and refused when tau = 31."""
    # G0 = rank 0: e0 = 60, e2 = 50, e4 = 50;  G1 = rank 1: e1 = 30, e3 = 35, e5 = 35
    g = golden("swap_example")
    e2r = np.array([0, 1, 0, 1, 0, 1], np.int32)
    cnt = np.array([g["e0_tokens"], g["e1_tokens"], 50, 35, 50, 35], np.int32)
    assert list(np.bincount(e2r, weights=cnt)) == g["loads_before"]
    prob, keep = _prob(oracle_mod, 1, 6, 2, 2, 1, e2r=e2r)
    new, swaps = oracle_mod.swap_plan(prob, cnt, 30)
    a, b, x, y, old, best = swaps[0, 0]
    assert (a, b, x, y, old, best) == (0, 1, 0, 1, max(g["loads_before"]), max(g["loads_after"]))
    assert list(new) == [1, 0, 0, 1, 0, 1]
    loads = np.bincount(new, weights=cnt, minlength=2)
    assert list(loads) == g["loads_after"]
    new31, _ = oracle_mod.swap_plan(prob, cnt, 31)
    assert np.array_equal(new31, e2r)


def test_swap_plan_is_the_best_single_exchange(oracle_mod):
    """Brute force on small random hosts: the chosen exchange attains the
    smallest pair maximum, pairs are heaviest-with-lightest, and only accepted
    pairs move experts."""
    rng = np.random.default_rng(4)
    for trial in range(40):
        P = int(rng.choice([2, 3, 4, 6]))
        H = int(rng.integers(1, 4))
        R = P * H
        per = int(rng.integers(1, 4))
        E = R * per
        e2r = rng.permutation(np.repeat(np.arange(R), per)).astype(np.int32)
        cnt = rng.integers(0, 200, E).astype(np.int32)
        tau = int(rng.integers(0, 40))
        prob, keep = _prob(oracle_mod, 1, E, R, P, 1, e2r=e2r)
        new, swaps = oracle_mod.swap_plan(prob, cnt, tau)
        load = np.bincount(e2r, weights=cnt, minlength=R).astype(np.int64)
        moved = set()
        for hh in range(H):
            order = sorted(range(hh * P, (hh + 1) * P), key=lambda r: (-load[r], r))
            for i in range(P // 2):
                a, b, x, y, old, best = swaps[hh, i]
                assert (a, b) == (order[i], order[P - 1 - i])
                assert old == max(load[a], load[b])
                cands = [(max(load[a] - cnt[xx] + cnt[yy], load[b] - cnt[yy] + cnt[xx]), xx, yy)
                         for xx in np.nonzero(e2r == a)[0] for yy in np.nonzero(e2r == b)[0]]
                m, bx, by = min(cands)
                assert (best, x, y) == (m, bx, by)
                if old - best >= max(tau, 1):
                    assert new[x] == b and new[y] == a
                    moved |= {x, y}
        for e in range(E):
            if e not in moved:
                assert new[e] == e2r[e]


# ------------------------------------------------ Mode 2 relay on one buffer

def test_relay_layout_and_dispatch(oracle_mod):
    """Relay rows: one per (token, host) with the mask bit, host segments at
    host_offset in ascending token order; their number is the per-host
    de-duplicated count (Mode 2 network copies plus one local copy per token
    whose experts include its own host).  Two-hop dispatch equals the flat
    dispatch byte for byte."""
    w = mw.Workload("rel", T=150, h=64, k=4, E=24, R=6, P=2, R_src=3)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=w.R_src)
    lay = oracle_mod.layout(prob, ids)
    rp = oracle_mod.relay_layout(prob, ids)
    assert np.array_equal(rp >= 0, lay["host_mask"].astype(bool))
    for hh in range(w.H):
        col = rp[:, hh][rp[:, hh] >= 0]
        assert np.array_equal(col, lay["host_offset"][hh] + np.arange(lay["host_count"][hh]))
    st = oracle_mod.stats(prob, ids)
    own = np.arange(w.T) // (w.T // w.R_src) // w.P
    local = lay["host_mask"][np.arange(w.T), own].sum()
    assert (rp >= 0).sum() == st["sum_mode2_copies"] + local
    x = mw.gen_x_bf16(w)
    relay, _, recv, _ = oracle_mod.relay_dispatch(prob, ids, lay["pos"], rp, x)
    assert np.array_equal(recv, oracle_mod.dispatch(prob, lay["pos"], x))
    for hh in range(w.H):
        toks = np.nonzero(rp[:, hh] >= 0)[0]
        assert np.array_equal(relay[rp[toks, hh]], x[toks])


def test_relay_combine_exact_when_no_rounding(oracle_mod):
    """With small-integer expert outputs and unit weights every partial and
    sum is exact, so two-hop combine equals flat combine bit for bit."""
    w = mw.Workload("rel2", T=100, h=32, k=4, E=16, R=8, P=2, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    rp = oracle_mod.relay_layout(prob, ids)
    y = mw.f32_to_bf16_bits(np.random.default_rng(3).integers(-20, 20, (w.slots, w.h)).astype(np.float32))
    ones = np.ones((w.T, w.k), np.float32)
    _, out = oracle_mod.relay_combine(prob, ids, lay["pos"], rp, y, ones)
    assert np.array_equal(out, oracle_mod.combine(prob, lay["pos"], y, ones))


def test_relay_combine_error_bound(oracle_mod):
    """Two roundings to bf16 (the partial and the result) plus fp32 sums:
    |out - exact| <= 2^-8 |exact| + 2^-8 sum_H |partial_H| + fp32 terms."""
    w = mw.Workload("rel3", T=80, h=256, k=8, E=32, R=8, P=2, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    rp = oracle_mod.relay_layout(prob, ids)
    y = mw.gen_y_host(w)
    g = mw.gen_gates(w)
    _, out = oracle_mod.relay_combine(prob, ids, lay["pos"], rp, y, g)
    terms = g.astype(np.float64)[:, :, None] * mw.bf16_bits_to_f32(y).astype(np.float64)[lay["pos"]]
    exact = terms.sum(axis=1)
    host = (ids // (w.E // w.R)) // w.P
    part = np.stack([np.where((host == hh)[:, :, None], terms, 0).sum(axis=1) for hh in range(w.H)])
    bound = (2.0 ** -8 * np.abs(exact) + 2.0 ** -8 * np.abs(part).sum(axis=0)
             + 2 * w.k * 2.0 ** -24 * np.abs(terms).sum(axis=1))
    got = mw.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound * (1 + 1e-9))


def test_relay_combine_one_host_is_flat(oracle_mod):
    """With every rank on one host there is one partial per token, equal to the
    flat combine; the final sum of that single partial adds nothing, so the
    two-hop result equals the flat combine bit for bit at any values."""
    w = mw.Workload("rel4", T=90, h=128, k=6, E=32, R=8, P=8, R_src=1)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h)
    lay = oracle_mod.layout(prob, ids)
    rp = oracle_mod.relay_layout(prob, ids)
    assert np.array_equal(rp[:, 0], np.arange(w.T))
    y, g = mw.gen_y_host(w), mw.gen_gates(w)
    partial, out = oracle_mod.relay_combine(prob, ids, lay["pos"], rp, y, g)
    flat = oracle_mod.combine(prob, lay["pos"], y, g)
    assert np.array_equal(partial, flat) and np.array_equal(out, flat)


def test_relay_dispatch_fp8_scales_travel(oracle_mod):
    """fp8 rows take their per-128-column scales through both hops."""
    w = mw.Workload("rel5", T=60, h=256, k=4, E=16, R=8, P=4, R_src=2, dtype="fp8")
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, R_src=w.R_src, elem_bytes=1)
    lay = oracle_mod.layout(prob, ids)
    rp = oracle_mod.relay_layout(prob, ids)
    x, xs = mw.gen_x_fp8(w)
    relay, rs, recv, rcs = oracle_mod.relay_dispatch(prob, ids, lay["pos"], rp, x, xs)
    flat = lay["recv_src"] // w.k
    assert np.array_equal(recv, x[flat]) and np.array_equal(rcs, xs[flat])
    toks = np.nonzero(rp >= 0)[0]
    assert np.array_equal(rs[rp[rp >= 0]], xs[toks])


# ------------------------------------------------ per-expert-group overlap

@pytest.mark.parametrize("E,R,G,custom", [(128, 16, 2, False), (256, 32, 4, False), (48, 12, 4, True),
                                          (64, 8, 1, False), (30, 6, 4, True)])
def test_expert_groups_split_every_rank(oracle_mod, E, R, G, custom):
    """Every rank's experts, in ascending order, form G contiguous runs whose
    sizes differ by at most one (no run empty when the rank has >= G experts)."""
    rng = np.random.default_rng(E + G)
    e2r = rng.integers(0, R, size=E).astype(np.int32) if custom else None
    prob, keep = _prob(oracle_mod, 64, E, R, 2, 2, e2r=e2r)
    grp = oracle_mod.expert_groups(prob, G)
    rank = e2r if custom else np.arange(E) // (E // R)
    for r in range(R):
        seq = grp[np.nonzero(rank == r)[0]]
        if len(seq) == 0:
            continue
        assert np.all(np.diff(seq) >= 0) and seq.min() >= 0 and seq.max() < G
        sizes = np.bincount(seq, minlength=G)
        if len(seq) >= G:
            assert sizes.min() >= 1
        assert sizes.max() - sizes.min() <= 1


def _group_case(oracle_mod, T=120, h=64, k=8, E=64, R=8, P=4, G=2, dtype="bf16", sort_by_group=False, seed=0):
    w = mw.Workload("peo", T=T, h=h, k=k, E=E, R=R, P=P, R_src=1, dtype=dtype, seed=seed)
    ids = mw.gen_ids(w)
    prob, keep = _prob(oracle_mod, w.T, w.E, w.R, w.P, w.k, h=w.h, elem_bytes=1 if dtype == "fp8" else 2)
    grp = oracle_mod.expert_groups(prob, G)
    if sort_by_group:
        order = np.argsort(grp[ids], axis=1, kind="stable")
        ids = np.take_along_axis(ids, order, axis=1)
    lay = oracle_mod.layout(prob, ids)
    return w, ids, prob, keep, grp, lay


@pytest.mark.parametrize("G", [1, 2, 4])
def test_group_dispatch_partitions_flat_dispatch(oracle_mod, G):
    """The G group dispatches write disjoint receive rows whose union is the
    flat dispatch (bf16 and fp8 with scales)."""
    for dtype in ("bf16", "fp8"):
        w, ids, prob, keep, grp, lay = _group_case(oracle_mod, G=G, dtype=dtype, h=256)
        if dtype == "fp8":
            x, xs = mw.gen_x_fp8(w)
            flat = (oracle_mod.dispatch(prob, lay["pos"], x, xs))
        else:
            x, xs = mw.gen_x_bf16(w), None
            flat = (oracle_mod.dispatch(prob, lay["pos"], x),)
        written = np.zeros(w.slots, np.int32)
        recv = rs = None
        for g in range(G):
            before = None if recv is None else recv.copy()
            recv, rs = oracle_mod.dispatch_group(prob, ids, lay["pos"], grp, g, x, xs, recv, rs)
            rows = lay["pos"][grp[ids] == g]
            written[rows] += 1
            if before is not None:   # rows of other groups untouched
                others = np.setdiff1d(np.arange(w.slots), rows)
                assert np.array_equal(recv[others][written[others] == 0], before[others][written[others] == 0])
        assert np.all(written == 1)
        assert np.array_equal(recv, flat[0])
        if dtype == "fp8":
            assert np.array_equal(rs, flat[1])


def test_group_combine_one_group_is_flat(oracle_mod):
    w, ids, prob, keep, grp, lay = _group_case(oracle_mod, G=1, h=128)
    y, g = mw.gen_y_host(w), mw.gen_gates(w)
    accs, out = oracle_mod.combine_groups(prob, ids, lay["pos"], grp, 1, y, g)
    assert accs == [] and np.array_equal(out, oracle_mod.combine(prob, lay["pos"], y, g))


@pytest.mark.parametrize("G", [2, 4])
def test_group_combine_in_slot_order_is_flat(oracle_mod, G):
    """When every token lists its experts group by group, the group-major
    chain is the ascending-slot chain: bit-exact equal to the flat combine."""
    w, ids, prob, keep, grp, lay = _group_case(oracle_mod, G=G, h=128, sort_by_group=True)
    y, g = mw.gen_y_host(w), mw.gen_gates(w)
    accs, out = oracle_mod.combine_groups(prob, ids, lay["pos"], grp, G, y, g)
    assert np.array_equal(out, oracle_mod.combine(prob, lay["pos"], y, g))
    # the fp32 accumulator after group 0 holds the sum of the group-0 terms
    # only, within the error of an fp32 chain of k terms
    terms = g.astype(np.float64)[:, :, None] * mw.bf16_bits_to_f32(y).astype(np.float64)[lay["pos"]]
    in0 = (grp[ids] == 0)[:, :, None]
    exact0 = np.where(in0, terms, 0.0).sum(axis=1)
    bound0 = w.k * 2.0 ** -24 * np.abs(np.where(in0, terms, 0.0)).sum(axis=1)
    assert np.all(np.abs(accs[0].astype(np.float64) - exact0) <= bound0)


@pytest.mark.parametrize("G", [2, 4])
def test_group_combine_exact_and_bounded(oracle_mod, G):
    """Any slot order: integer data with unit weights is exact (equal to the
    flat combine); random data is within the fp32-chain + bf16 bound of the
    exact sum."""
    w, ids, prob, keep, grp, lay = _group_case(oracle_mod, G=G, h=64)
    yi = mw.f32_to_bf16_bits(np.random.default_rng(4).integers(-30, 30, (w.slots, w.h)).astype(np.float32))
    ones = np.ones((w.T, w.k), np.float32)
    _, out = oracle_mod.combine_groups(prob, ids, lay["pos"], grp, G, yi, ones)
    assert np.array_equal(out, oracle_mod.combine(prob, lay["pos"], yi, ones))
    y, g = mw.gen_y_host(w), mw.gen_gates(w)
    _, out = oracle_mod.combine_groups(prob, ids, lay["pos"], grp, G, y, g)
    terms = g.astype(np.float64)[:, :, None] * mw.bf16_bits_to_f32(y).astype(np.float64)[lay["pos"]]
    exact = terms.sum(axis=1)
    bound = 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * w.k * 2.0 ** -24 * np.abs(terms).sum(axis=1)
    got = mw.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound)
