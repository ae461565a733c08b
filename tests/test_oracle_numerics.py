"""Pins for the oracle's number formats, payload movement and combine (CPU only)."""
import math

import numpy as np
import pytest
import torch

import workloads
from workloads import from_bf16_bits, to_bf16_bits

# ---------------------------------------------------------------- bf16


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(3)
    f = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4000),
                        # exact ties: low 16 bits 0x8000, both parities of bit 16
                        (np.arange(200, dtype=np.uint32) << 16 | 0x3F800000 | 0x8000).view(np.float32)])
    want = to_bf16_bits(f.astype(np.float32))
    got = np.array([orc.f32_to_bf16(v) for v in f], np.uint16)
    np.testing.assert_array_equal(got, want)
    b = rng.integers(0, 1 << 16, 3000).astype(np.uint16)
    b = b[~np.isnan(from_bf16_bits(b))]
    np.testing.assert_array_equal(np.array([orc.bf16_to_f32(v) for v in b], np.float32), from_bf16_bits(b))


# ---------------------------------------------------------------- OCP FP8 E4M3

# (code, value) pairs from the OCP 8-bit floating point specification (v1.0), E4M3 column:
# bias 7, max normal S.1111.110 = 448, min normal 2^-6, subnormals m * 2^-9, NaN S.1111.111.
def _known_values():
    out = []
    for line in open(__file__.replace("test_oracle_numerics.py", "golden/e4m3_known_values.txt")):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


def test_e4m3_decode_known_values(orc):
    kv = _known_values()
    assert len(kv) >= 15
    for c, v in kv:
        got = orc.e4m3_decode(c)
        if math.isnan(v):
            assert math.isnan(got), hex(c)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(c), got, v)


def test_e4m3_decode_matches_torch_all_codes(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def _finite_table():
    """All finite E4M3 codes with their values, decoded by torch (not by the oracle)."""
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    keep = ~np.isnan(vals)
    return np.arange(256)[keep], vals[keep]


def _brute_encode(v, codes, vals):
    """Nearest finite code by exhaustive search; ties to the code with even mantissa;
    beyond +-448 saturate. Signed zero keeps its sign."""
    if v >= 448:
        return 0x7E
    if v <= -448:
        return 0xFE
    same_sign = (codes & 0x80) == (0x80 if math.copysign(1, v) < 0 else 0)
    c, x = codes[same_sign], vals[same_sign]
    dist = np.abs(x - v)
    best = dist.min()
    cand = c[dist == best]
    if len(cand) > 1:
        cand = cand[(cand & 1) == 0]
    return int(cand[0])


def test_e4m3_encode_matches_exhaustive_nearest(orc):
    codes, vals = _finite_table()
    pos = np.sort(np.unique(vals[vals >= 0]))
    mids = (pos[:-1] + pos[1:]) / 2           # exact ties, all representable in fp32
    probe = [float(np.float32(m)) for m in mids]
    probe += [float(np.nextafter(np.float32(m), np.float32(np.inf))) for m in mids]
    probe += [float(np.nextafter(np.float32(m), np.float32(-np.inf))) for m in mids]
    probe += list(pos) + [447.9, 448.0, 448.5, 460.0, 464.0, 470.0, 1e6, 2.0 ** -10, 2.0 ** -12, 0.0]
    rng = np.random.default_rng(9)
    probe += list(rng.uniform(-500, 500, 3000).astype(np.float32).astype(float))
    probe += list((rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 6, 3000)).astype(np.float32).astype(float))
    probe += [-p for p in probe[:500]]
    for v in probe:
        assert orc.e4m3_encode(v) == _brute_encode(v, codes, vals), v


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-447, 447, 5000), rng.standard_normal(5000) * 2.0 ** -7]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in v], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_decode_identity_on_finite_codes(orc):
    for c in range(256):
        v = orc.e4m3_decode(c)
        if not math.isnan(v):
            assert orc.e4m3_encode(v) == c, hex(c)


# ---------------------------------------------------------------- block-scaled quantisation


def test_quantize_fp8_scale_and_bound(orc):
    rng = np.random.default_rng(5)
    H = 512
    xf = (rng.standard_normal((6, H)) * np.exp(rng.uniform(-6, 6, (6, 1)))).astype(np.float32)
    xf[2, 128:256] = 0.0                        # an all-zero block -> scale 1, codes 0
    x = to_bf16_bits(xf)
    q = orc.quantize_fp8(x)
    assert q.shape == (6, H + 4 * (H // 128))
    xv = from_bf16_bits(x)
    codes, vals = _finite_table()
    lut = np.full(256, np.nan)
    lut[codes] = vals
    for r in range(6):
        sc = q[r, H:].copy().view(np.float32)
        for b in range(H // 128):
            blk = xv[r, b * 128:(b + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            want = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
            assert sc[b] == want
            deq = lut[q[r, b * 128:(b + 1) * 128]] * float(sc[b])
            # E4M3 keeps 3 mantissa bits: relative error <= 2^-4, absolute 2^-10 * scale near 0
            err = np.abs(deq - blk.astype(np.float64))
            assert (err <= 2.0 ** -4 * np.abs(blk) + 2.0 ** -10 * float(sc[b])).all()
            assert np.abs(deq).max() <= 448.0 * float(sc[b]) * (1 + 2.0 ** -20)
    assert (q[2, 128:256] == 0).all() and q[2, H + 4:H + 8].view(np.float32)[0] == 1.0


def test_expert_dequant_definition(orc):
    rng = np.random.default_rng(6)
    N, L, cap, H = 2, 2, 3, 256
    exq = rng.integers(0, 256, (N, L, cap, H)).astype(np.uint8)
    exq[(exq & 0x7F) == 0x7F] = 0x11              # no NaN codes
    exs = rng.uniform(0.001, 2.0, (N, L, cap, H // 128)).astype(np.float32)
    lay = {"ecnt": np.array([[3, 1], [0, 2]], np.int32)}
    ey = orc.expert_dequant(N, L, cap, H, exq, exs, lay)
    codes, vals = _finite_table()
    lut = np.zeros(256)
    lut[codes] = vals
    prod = (lut[exq].astype(np.float32) * np.repeat(exs, 128, axis=-1)).astype(np.float32)  # one fp32 rounding
    want = to_bf16_bits(prod)
    for d in range(N):
        for l in range(L):
            n = lay["ecnt"][d, l]
            np.testing.assert_array_equal(ey[d, l, :n], want[d, l, :n])
            assert (ey[d, l, n:] == 0).all()


# ---------------------------------------------------------------- payload movement and combine


def _fwd(orc, wl, w=None, idx=None, x=None):
    inp = workloads.make_inputs(wl)
    if w is not None:
        inp["w"] = w
    if idx is not None:
        inp["idx"] = idx
    if x is not None:
        inp["x"] = x
    r = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    return inp, r


SMALL = [
    workloads.config(0),
    workloads.Workload("small-a", 4, 9, 256, 12, 3, "bf16", "uniform", 21),
    workloads.Workload("small-zipf", 3, 11, 128, 9, 4, "bf16", "zipf", 22),
    workloads.Workload("small-skew", 4, 6, 128, 16, 4, "bf16", "skew0", 23),
    workloads.Workload("small-fp8", 4, 5, 512, 8, 2, "fp8", "uniform", 24),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_payload_rows_are_the_routed_tokens(orc, wl):
    inp, r = _fwd(orc, wl)
    lay = r["layout"]
    N, T, R, H = wl.N, wl.T, wl.R, wl.H
    xrows = r["xq"] if wl.payload == "fp8" else inp["x"].view(np.uint8)
    xrows = xrows.reshape(N * T, -1)
    ss, rs = lay["slot_src"], lay["recv_src"]
    for d in range(N):
        for i in range(lay["rtot"][d]):                 # receive row i holds its pair's token
            q = rs[d, i]
            np.testing.assert_array_equal(r["recv"][d, i], xrows[q // R])
    for d in range(N):
        for l in range(wl.L):
            for j in range(min(lay["ecnt"][d, l], lay["cap"])):   # grouped row j holds its pair's token
                q = ss[d, l, j]
                if wl.payload == "fp8":
                    np.testing.assert_array_equal(r["exq"][d, l, j], xrows[q // R][:H])
                    np.testing.assert_array_equal(r["exs"][d, l, j].view(np.uint8), xrows[q // R][H:])
                else:
                    np.testing.assert_array_equal(r["ex"][d, l, j].view(np.uint8), xrows[q // R])
    # combine send returns to every pair the expert output of its own token
    ey_tok = r["ey"] if wl.payload == "fp8" else None
    for s in range(N):
        for t in range(T):
            for k in range(R):
                p = lay["pos"][s, t, k]
                if wl.payload == "bf16":
                    np.testing.assert_array_equal(r["crecv"][s, p], inp["x"][s, t])
                else:
                    e = inp["idx"][s, t, k]
                    d, l = e // wl.L, e % wl.L
                    np.testing.assert_array_equal(r["crecv"][s, p], ey_tok[d, l, lay["slot"][s, t, k]])


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_round_trip_exact_with_equal_power_of_two_weights(orc, R):
    """Identity experts, w = 1/R: every partial sum j*x/R of a bf16 x is exact in fp32,
    so dispatch -> identity -> combine returns x bit for bit."""
    wl = workloads.Workload("rt", 4, 7, 256, 16, R, "bf16", "uniform", 30 + R)
    w = np.full((wl.N, wl.T, R), 1.0 / R, np.float32)
    inp, r = _fwd(orc, wl, w=w)
    np.testing.assert_array_equal(r["out"], inp["x"])


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_round_trip_softmax_within_tolerance(orc, wl):
    inp, r = _fwd(orc, wl)
    x = from_bf16_bits(inp["x"]).astype(np.float64)
    if wl.payload == "fp8":
        # the identity expert returns the dequantised token, so combine returns it too
        codes, vals = _finite_table()
        lut = np.zeros(256)
        lut[codes] = vals
        H = wl.H
        xq = r["xq"].reshape(wl.N, wl.T, -1)
        sc = xq[..., H:].copy().view(np.float32)
        deq = lut[xq[..., :H]] * np.repeat(sc, 128, axis=-1)
        assert np.abs(deq - x).max() <= 2.0 ** -4 * np.abs(x).max()
        x = from_bf16_bits(to_bf16_bits(deq.astype(np.float32))).astype(np.float64)
    tol = 2.0 ** -7 * np.abs(x).max()
    assert np.abs(from_bf16_bits(r["out"]) - x).max() <= tol
    assert np.abs(r["out64"] - x).max() <= 2.0 ** -20 * np.abs(x).max()


def test_combine_sum_against_exact_fsum(orc):
    wl = SMALL[1]
    inp, r = _fwd(orc, wl)
    lay = r["layout"]
    N, T, R, H = wl.N, wl.T, wl.R, wl.H
    cre = from_bf16_bits(r["crecv"]).astype(np.float64)
    w = inp["w"].astype(np.float64)
    for s in range(N):
        for t in range(T):
            terms = np.stack([w[s, t, k] * cre[s, lay["pos"][s, t, k]] for k in range(R)])  # exact products
            for h in range(0, H, 7):
                exact = math.fsum(terms[:, h])
                mag = float(np.abs(terms[:, h]).sum())
                assert abs(r["out64"][s, t, h] - exact) <= R * 2.0 ** -52 * mag
                # fp32 accumulation then one bf16 rounding: within a bf16 ulp of the exact sum
                o = float(from_bf16_bits(np.array([r["out"][s, t, h]], np.uint16))[0])
                assert abs(o - exact) <= 2.0 ** -8 * abs(exact) + R * 2.0 ** -23 * mag + 1e-30


def test_combine_skips_dropped_and_invalid_pairs(orc):
    wl = workloads.Workload("drop", 2, 4, 128, 4, 2, "bf16", "uniform", 40, cap=3)
    idx = np.array([[[0, 1], [0, 2], [0, 3], [0, -1]], [[0, 1], [2, 3], [5, 1], [1, 0]]], np.int32)
    w = np.full((2, 4, 2), 0.5, np.float32)
    inp, r = _fwd(orc, wl, idx=idx, w=w)
    lay = r["layout"]
    assert lay["status"] == orc.BIT_EXPERT_RANGE | orc.BIT_CAPACITY
    x = from_bf16_bits(inp["x"])
    out = from_bf16_bits(r["out"])
    # the combine rows of dropped pairs are never written; fill them with 1.0 so that a
    # combine which read them would differ
    _, crecv1 = orc.combine_send(wl.N, wl.T, wl.E, wl.R, lay["cap"], wl.H, r["ey"], lay, fill=0x3F80)
    out1, _ = orc.combine_recv(wl.N, wl.T, wl.R, wl.H, crecv1, w, lay)
    for o in (out, from_bf16_bits(out1)):
        for s in range(2):
            for t in range(4):
                keep = [(k) for k in range(2) if lay["pos"][s, t, k] >= 0 and lay["slot"][s, t, k] >= 0]
                want = sum(np.float32(0.5) * x[s, t] for _ in keep) if keep else np.zeros(wl.H, np.float32)
                np.testing.assert_array_equal(o[s, t], from_bf16_bits(to_bf16_bits(np.asarray(want, np.float32))))


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_run_step_equals_forward(orc, wl):
    inp = workloads.make_inputs(wl)
    r = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    b = orc.alloc_step(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload)
    st = orc.run_step(b, inp["x"], inp["idx"], inp["w"])
    assert st == r["layout"]["status"]
    np.testing.assert_array_equal(b["out"], r["out"])
    np.testing.assert_array_equal(b["out64"], r["out64"])


# ---------------------------------------------------------------- combine with expert-side partial sums


def _partial(orc, wl, inp, r):
    L = wl.L
    lay = r["layout"]
    return orc.combine_partial(wl.N, wl.T, wl.E, wl.R, wl.cap, wl.H, r["ey"], inp["w"], inp["idx"], lay,
                               fill=0x7FFF)


@pytest.mark.parametrize("wl", [SMALL[3], workloads.config(4).replace(T=24, H=256, seed=44),
                                workloads.Workload("r1", 4, 9, 256, 12, 1, "bf16", "uniform", 45)],
                         ids=["skew-small", "skew-cfg4-shape", "R1"])
def test_partial_combine_equals_canonical_with_one_group_per_token(orc, wl):
    """When all of a token's experts sit on one rank there is one partial per token: it is
    the canonical fp32 sum rounded once, so both combines agree bit for bit."""
    inp, r = _fwd(orc, wl)
    cpart, out = _partial(orc, wl, inp, r)
    np.testing.assert_array_equal(out, r["out"])
    np.testing.assert_array_equal(cpart[:, :, 0], r["out"])
    if cpart.shape[2] > 1:
        assert (cpart[:, :, 1:] == 0x7FFF).all()          # rows past the groups are untouched


@pytest.mark.parametrize("wl", SMALL[:3] + [workloads.config(1).replace(T=6, H=256, seed=46)], ids=lambda w: w.name)
def test_partial_combine_within_tolerance_and_restated(orc, wl):
    inp, r = _fwd(orc, wl)
    cpart, out = _partial(orc, wl, inp, r)
    x = from_bf16_bits(inp["x"]).astype(np.float64)
    # one bf16 rounding per group plus one of the sum: within 2^-7 max|x| of the exact sum
    assert np.abs(from_bf16_bits(out) - r["out64"]).max() <= 2.0 ** -7 * np.abs(x).max()
    # independent restatement: group pairs by owner rank with numpy, fp32 scalar arithmetic
    lay = r["layout"]
    ey = from_bf16_bits(r["ey"])
    N, T, R, L = wl.N, wl.T, wl.R, wl.L
    for s in range(N):
        for t in range(T):
            ks = [k for k in range(R) if lay["slot"][s, t, k] >= 0]
            owners = sorted({int(inp["idx"][s, t, k]) // L for k in ks})
            total = np.zeros(wl.H, np.float32)
            for j, d in enumerate(owners):
                acc = np.zeros(wl.H, np.float32)
                for k in ks:
                    e = int(inp["idx"][s, t, k])
                    if e // L == d:
                        acc = (acc + np.float32(inp["w"][s, t, k]) * ey[d, e % L, lay["slot"][s, t, k]]).astype(np.float32)
                p = to_bf16_bits(acc)
                np.testing.assert_array_equal(cpart[s, t, j], p)
                total = (total + from_bf16_bits(p)).astype(np.float32)
            np.testing.assert_array_equal(out[s, t], to_bf16_bits(total))


# ---------------------------------------------------------------- combine with distinct expert outputs

def _random_expert_rows(wl, cap, seed):
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal((wl.N, wl.L, cap, wl.H)).astype(np.float32))


DISTINCT = [SMALL[1], SMALL[2], workloads.Workload("dup-cap", 3, 10, 128, 6, 4, "bf16", "uniform", 47, cap=7)]


@pytest.mark.parametrize("wl", DISTINCT, ids=lambda w: w.name)
def test_combine_with_distinct_expert_outputs_restated(orc, wl):
    """Every expert returns its own rows, so each (token, expert) pair brings a different row:
    combine must pair weight k with the row of expert idx[k] at slot[k]. Restated per pair
    from idx, slot and the weights alone (fp32, k ascending, separate rounding), bit for bit;
    the fp64 variant against an exact sum."""
    inp = workloads.make_inputs(wl)
    if wl.name == "dup-cap":   # duplicates within tokens, bad ids, and capacity drops
        rng = np.random.default_rng(48)
        inp["idx"] = rng.integers(0, wl.E, size=(wl.N, wl.T, wl.R)).astype(np.int32)
        inp["idx"][0, 2, 1] = -1
    lay = orc.layout(wl.N, wl.T, wl.E, wl.R, wl.cap, inp["idx"])
    cap, L = lay["cap"], wl.L
    ey = _random_expert_rows(wl, cap, 49)
    csend, crecv = orc.combine_send(wl.N, wl.T, wl.E, wl.R, cap, wl.H, ey, lay)
    out, out64 = orc.combine_recv(wl.N, wl.T, wl.R, wl.H, crecv, inp["w"], lay)
    y = from_bf16_bits(ey)
    for s in range(wl.N):
        for t in range(wl.T):
            acc = np.zeros(wl.H, np.float32)
            terms = []
            for k in range(wl.R):
                e, j = int(inp["idx"][s, t, k]), int(lay["slot"][s, t, k])
                if 0 <= e < wl.E and j >= 0:
                    row = y[e // L, e % L, j]
                    acc = (acc + (np.float32(inp["w"][s, t, k]) * row).astype(np.float32)).astype(np.float32)
                    terms.append(np.float64(inp["w"][s, t, k]) * row.astype(np.float64))
            np.testing.assert_array_equal(out[s, t], to_bf16_bits(acc), err_msg=f"token ({s},{t})")
            if terms:
                exact = np.array([math.fsum(c) for c in np.stack(terms).T])
                assert np.abs(out64[s, t] - exact).max() <= wl.R * 2.0 ** -52 * np.abs(np.stack(terms)).sum(0).max()


@pytest.mark.parametrize("wl", DISTINCT[:2], ids=lambda w: w.name)
def test_partial_combine_with_distinct_expert_outputs_restated(orc, wl):
    """Sender-side partial combine with per-expert rows: groups by owner rank ascending,
    weights paired with their own expert's row, restated per pair."""
    inp = workloads.make_inputs(wl)
    lay = orc.layout(wl.N, wl.T, wl.E, wl.R, wl.cap, inp["idx"])
    cap, L = lay["cap"], wl.L
    ey = _random_expert_rows(wl, cap, 50)
    cpart, out = orc.combine_partial(wl.N, wl.T, wl.E, wl.R, cap, wl.H, ey, inp["w"], inp["idx"], lay, fill=0x7FFF)
    y = from_bf16_bits(ey)
    for s in range(wl.N):
        for t in range(wl.T):
            ks = [k for k in range(wl.R) if lay["slot"][s, t, k] >= 0]
            owners = sorted({int(inp["idx"][s, t, k]) // L for k in ks})
            total = np.zeros(wl.H, np.float32)
            for jg, d in enumerate(owners):
                acc = np.zeros(wl.H, np.float32)
                for k in ks:
                    e = int(inp["idx"][s, t, k])
                    if e // L == d:
                        acc = (acc + (np.float32(inp["w"][s, t, k]) * y[d, e % L, lay["slot"][s, t, k]])
                               .astype(np.float32)).astype(np.float32)
                np.testing.assert_array_equal(cpart[s, t, jg], to_bf16_bits(acc))
                total = (total + from_bf16_bits(to_bf16_bits(acc))).astype(np.float32)
            np.testing.assert_array_equal(out[s, t], to_bf16_bits(total))
