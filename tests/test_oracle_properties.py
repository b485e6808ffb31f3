"""Property checks of the oracle over random small problems (hypothesis).

Each property follows from the definitions alone, so it pins the oracle
against something other than itself: the layout's counts, scans, bijection and
inverse; the host mask against the slots' hosts; the relay rows against the
mask; the expert groups against the placement; and a combine whose result is
exact (a single nonzero term, or all weights zero).
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import moe_workloads as mw  # noqa: E402


@st.composite
def problems(draw):
    P = draw(st.sampled_from([1, 2, 4]))
    H = draw(st.integers(1, 4))
    R = P * H
    custom = draw(st.booleans())
    per = draw(st.integers(1, 4))
    E = R * per
    k = draw(st.integers(1, min(E, 6)))
    T = draw(st.integers(0, 40))
    seed = draw(st.integers(0, 10_000))
    rng = np.random.default_rng(seed)
    ids = np.array([rng.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
    e2r = rng.integers(0, R, size=E).astype(np.int32) if custom else None
    return dict(T=T, E=E, R=R, P=P, k=k, ids=ids, e2r=e2r, seed=seed)


def _mk(oracle, p, h=16):
    return oracle.make_problem(p["T"], h, p["k"], p["E"], p["R"], p["P"], 1, 2, 128, p["e2r"], None)


def _rank(p):
    return (np.asarray(p["e2r"]) if p["e2r"] is not None else np.arange(p["E"]) // (p["E"] // p["R"]))


@settings(max_examples=150, deadline=None)
@given(problems())
def test_layout_properties(oracle_mod, p):
    prob, keep = _mk(oracle_mod, p)
    lay = oracle_mod.layout(prob, p["ids"])
    T, k, E, R, P = p["T"], p["k"], p["E"], p["R"], p["P"]
    ids = p["ids"]
    rank = _rank(p)
    assert lay["expert_count"].sum() == T * k
    assert np.array_equal(lay["expert_count"], np.bincount(ids.ravel(), minlength=E))
    assert np.array_equal(lay["rank_count"], np.bincount(rank[ids.ravel()], minlength=R) if T else np.zeros(R))
    assert np.array_equal(np.diff(lay["rank_offset"]), lay["rank_count"]) and lay["rank_offset"][0] == 0
    pos = lay["pos"].ravel()
    assert np.array_equal(np.sort(pos), np.arange(T * k))                    # a bijection
    assert np.array_equal(lay["recv_src"][pos], np.arange(T * k))            # its inverse
    # receive order: (rank, expert) ascending, then token ascending
    e_of_row = ids.ravel()[lay["recv_src"]]
    key = rank[e_of_row].astype(np.int64) * (E + 1) + e_of_row
    assert np.all(np.diff(key) >= 0)
    t_of_row = lay["recv_src"] // k
    same = np.diff(key) == 0
    assert np.all(np.diff(t_of_row)[same] > 0)
    # host mask and per-host counts
    H = R // P
    mask = np.zeros((T, H), np.uint8)
    for t in range(T):
        mask[t, rank[ids[t]] // P] = 1
    assert np.array_equal(lay["host_mask"], mask)
    assert np.array_equal(lay["host_count"], mask.sum(axis=0))


@settings(max_examples=100, deadline=None)
@given(problems())
def test_relay_and_group_properties(oracle_mod, p):
    prob, keep = _mk(oracle_mod, p)
    lay = oracle_mod.layout(prob, p["ids"])
    rp = oracle_mod.relay_layout(prob, p["ids"])
    assert np.array_equal(rp >= 0, lay["host_mask"].astype(bool))
    for hh in range(rp.shape[1] if rp.ndim == 2 else 0):
        col = rp[:, hh][rp[:, hh] >= 0]
        assert np.array_equal(col, lay["host_offset"][hh] + np.arange(len(col)))
    rank = _rank(p)
    for G in (1, 2, 3):
        grp = oracle_mod.expert_groups(prob, G)
        for r in range(p["R"]):
            seq = grp[np.nonzero(rank == r)[0]]
            if len(seq):
                assert seq[0] == 0 and np.all(np.diff(seq) >= 0) and seq[-1] == (len(seq) - 1) * G // len(seq)


@settings(max_examples=100, deadline=None)
@given(problems(), st.integers(0, 5))
def test_combine_single_term_is_exact(oracle_mod, p, j):
    """One nonzero weight per token: the fp32 chain is a single rounding of
    w * y, then bf16 RNE; all weights zero gives +0."""
    if p["T"] == 0:
        return
    h = 16
    prob, keep = _mk(oracle_mod, p, h)
    lay = oracle_mod.layout(prob, p["ids"])
    rng = np.random.default_rng(p["seed"])
    y = mw.f32_to_bf16_bits(rng.standard_normal((p["T"] * p["k"], h)).astype(np.float32))
    w = np.zeros((p["T"], p["k"]), np.float32)
    out0 = oracle_mod.combine(prob, lay["pos"], y, w)
    assert np.all(out0 == 0)
    jj = j % p["k"]
    w[:, jj] = rng.standard_normal(p["T"]).astype(np.float32)
    out = oracle_mod.combine(prob, lay["pos"], y, w)
    prod = (w[:, jj:jj + 1] * mw.bf16_bits_to_f32(y)[lay["pos"][:, jj]]).astype(np.float32)
    want = mw.f32_to_bf16_bits(prod)
    nz = prod != 0
    assert np.array_equal(out[nz], want[nz])
