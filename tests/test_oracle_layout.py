"""Pins for the oracle's layout: brute force, invariants and closed forms (CPU only)."""
import numpy as np
import pytest

import workloads
from tests import bruteforce
from tests.bruteforce import LAYOUT_KEYS


def _random_case(rng, allow_bad=True):
    N = int(rng.integers(1, 5))
    L = int(rng.integers(1, 5))
    E = N * L
    T = int(rng.integers(0, 9))
    R = int(rng.integers(1, 5))
    idx = rng.integers(0, E, size=(N, T, R)).astype(np.int32)   # duplicates allowed
    if allow_bad and T > 0 and rng.random() < 0.2:
        bad = rng.random(idx.shape) < 0.1
        idx[bad] = rng.choice(np.array([-1, E, E + 7, -100], np.int32), size=int(bad.sum()))
    cap = int(rng.integers(1, N * T + 1)) if (T > 0 and rng.random() < 0.3) else 0
    return N, T, E, R, cap, idx


def test_layout_matches_bruteforce_on_tiny_config(orc):
    wl = workloads.config(0)
    inp = workloads.make_inputs(wl)
    o = orc.layout(wl.N, wl.T, wl.E, wl.R, 0, inp["idx"])
    b = bruteforce.layout(wl.N, wl.T, wl.E, wl.R, 0, inp["idx"])
    for k in LAYOUT_KEYS:
        np.testing.assert_array_equal(o[k], b[k], err_msg=k)
    assert o["status"] == b["status"] == 0


def test_layout_matches_bruteforce_on_random_tiny_shapes(orc):
    rng = np.random.default_rng(12345)
    n_bad = n_cap = 0
    for _ in range(400):
        N, T, E, R, cap, idx = _random_case(rng)
        o = orc.layout(N, T, E, R, cap, idx)
        b = bruteforce.layout(N, T, E, R, cap, idx)
        for k in LAYOUT_KEYS:
            np.testing.assert_array_equal(o[k], b[k], err_msg=f"{k} N={N} T={T} E={E} R={R} cap={cap}")
        assert o["status"] == b["status"]
        n_bad += bool(o["status"] & orc.BIT_EXPERT_RANGE)
        n_cap += bool(o["status"] & orc.BIT_CAPACITY)
    assert n_bad > 5 and n_cap > 5   # the error paths were exercised


def _check_invariants(orc, N, T, E, R, cap, idx, o):
    L = E // N
    cap = cap if cap > 0 else N * T
    RB = N * T * max(R, L)
    valid = (idx >= 0) & (idx < E)
    nvalid = int(valid.sum())
    # every valid pair is received exactly once, within the N*T*max(R,E/N) bound
    assert int(o["rtot"].sum()) == nvalid
    assert (o["rtot"] <= RB).all()
    assert (o["ecnt"].sum(axis=1) == o["rtot"]).all()
    assert (o["cnt"].sum(axis=1) == valid.reshape(N, -1).sum(axis=1)).all()
    for s in range(N):
        p = o["pos"][s][valid[s]]
        assert sorted(p.tolist()) == list(range(p.size))   # send rows: a permutation
    ids = np.arange(N * T * R).reshape(N, T, R)
    # receive rows: every valid pair exactly once, padding -1
    rs = o["recv_src"]
    for d in range(N):
        assert (rs[d, o["rtot"][d]:] == -1).all()
    got = np.sort(rs[rs >= 0])
    np.testing.assert_array_equal(got, np.sort(ids[valid]))
    # grouped rows: every kept pair exactly once
    ss = o["slot_src"]
    kept = valid & (o["slot"] >= 0)
    np.testing.assert_array_equal(np.sort(ss[ss >= 0]), np.sort(ids[kept]))
    # distinct experts per token -> the tight bound N*T*min(R,E/N) holds too
    if T > 0 and valid.all() and all(len(set(r)) == R for r in idx.reshape(-1, R).tolist()):
        assert (o["rtot"] <= N * T * min(R, L)).all()
        assert (o["ecnt"] <= N * T).all()


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_layout_invariants_on_configs(orc, cfg):
    wl = workloads.config(cfg)
    inp = workloads.make_inputs(wl, with_x=False)
    o = orc.layout(wl.N, wl.T, wl.E, wl.R, 0, inp["idx"])
    assert o["status"] == 0
    _check_invariants(orc, wl.N, wl.T, wl.E, wl.R, 0, inp["idx"], o)


def test_layout_invariants_random(orc):
    rng = np.random.default_rng(7)
    for _ in range(200):
        N, T, E, R, cap, idx = _random_case(rng)
        o = orc.layout(N, T, E, R, cap, idx)
        _check_invariants(orc, N, T, E, R, cap, idx, o)


def test_layout_closed_form_skew(orc):
    """Every token routed to all E/N = R experts of rank 0: rank 0 receives N*T*R rows."""
    wl = workloads.config(4)
    N, T, E, R, L = wl.N, wl.T, wl.E, wl.R, wl.L
    idx = workloads.make_inputs(wl, with_x=False)["idx"]
    o = orc.layout(N, T, E, R, 0, idx)
    assert o["rtot"][0] == N * T * R == wl.RB          # the receive bound is met exactly
    assert (o["rtot"][1:] == 0).all()
    assert (o["ecnt"][0] == N * T).all() and (o["ecnt"][1:] == 0).all()
    for l in range(L):
        np.testing.assert_array_equal(o["eoff"][0, l], np.arange(N) * T)
    ss = o["slot_src"][0]                             # [L, cap]
    j = np.arange(N * T)
    s_of, t_of = ss // (T * R), (ss // R) % T
    for l in range(L):
        np.testing.assert_array_equal(s_of[l], j // T)
        np.testing.assert_array_equal(t_of[l], j % T)
        np.testing.assert_array_equal(idx.reshape(-1)[ss[l]], np.full(N * T, l))
    np.testing.assert_array_equal(o["roff"][0], np.arange(N) * T * R)
    assert (o["recv_src"][0] >= 0).all()


@pytest.mark.parametrize("N,T", [(4, 8), (8, 16), (3, 9)])
def test_layout_closed_form_rotation(orc, N, T):
    """R = 1, E = N, token t of rank s -> expert (s+t) mod N: a known all-to-all permutation."""
    s = np.arange(N)[:, None]
    t = np.arange(T)[None, :]
    idx = ((s + t) % N).astype(np.int32).reshape(N, T, 1)
    o = orc.layout(N, T, N, 1, 0, idx)
    P = T // N   # T is a multiple of N
    assert T % N == 0
    e = (s + t) % N
    np.testing.assert_array_equal(o["pos"][:, :, 0], e * P + t // N)
    np.testing.assert_array_equal(o["slot"][:, :, 0], s * P + t // N)
    np.testing.assert_array_equal(o["rrow"][:, :, 0], s * P + t // N)
    np.testing.assert_array_equal(o["roff"], np.tile(np.arange(N) * P, (N, 1)))
    np.testing.assert_array_equal(o["cnt"], np.full((N, N), P))
    np.testing.assert_array_equal(o["rtot"], np.full(N, T))


def test_layout_empty_and_degenerate(orc):
    # no tokens
    o = orc.layout(3, 0, 6, 2, 0, np.zeros((3, 0, 2), np.int32))
    assert o["status"] == 0 and o["rtot"].sum() == 0 and o["cnt"].sum() == 0
    # one rank holding every expert
    idx = np.array([[[0, 1], [1, 0], [1, 1]]], np.int32)
    o = orc.layout(1, 3, 2, 2, 0, idx)
    b = bruteforce.layout(1, 3, 2, 2, 0, idx)
    for k in LAYOUT_KEYS:
        np.testing.assert_array_equal(o[k], b[k])
    # expert 1 is routed 4 times but cap = N*T = 3: the 4th pair is dropped and flagged
    assert o["status"] == b["status"] == orc.BIT_CAPACITY
    assert o["slot"][0, 2, 1] == -1
