"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Nothing here re-types the oracle's formulas and compares them with themselves:
each check is a brute-force scalar expansion, a closed form, an invariant, a
special case reducing to a textbook result, or a number printed on a page.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O
from oracle import op_counts as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, B=2, H=3, d_c=16, d_rope=4, d_nope=6, d_v=5, S=9, lengths=None):
    cache = rng.standard_normal((B, S, d_c + d_rope))
    q_nope = rng.standard_normal((B, H, d_nope))
    q_rope = rng.standard_normal((B, H, d_rope))
    w_uk = 0.3 * rng.standard_normal((H, d_nope, d_c))
    w_uv = 0.3 * rng.standard_normal((H, d_v, d_c))
    if lengths is None:
        lengths = rng.integers(1, S + 1, size=B)
    lengths = np.asarray(lengths)
    positions = lengths - 1
    return dict(q_nope=q_nope, q_rope=q_rope, w_uk=w_uk, w_uv=w_uv, cache=cache,
                lengths=lengths, positions=positions)


# ---------------------------------------------------------------- O-I1: naive == absorbed
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_naive_equals_absorbed_fp64(seed):
    """Absorption is exact associativity (Multi-Head Latent Attention, 3.3: the
    absorbed and naive layers agree); in fp64 the two forms agree to 1e-10."""
    rng = np.random.default_rng(seed)
    case = _rand_case(rng, S=17)
    scale = 1 / math.sqrt(6 + 4)
    a = O.decode_absorbed(**case, scale=scale, base=10000.0)
    n = O.decode_naive(**case, scale=scale, base=10000.0)
    assert np.max(np.abs(a["o"] - n["o"])) <= 1e-10
    for pa, pn in zip(a["p"], n["p"]):
        assert np.max(np.abs(pa - pn)) <= 1e-12


def test_naive_equals_absorbed_v2lite_shapes():
    """Same at DeepSeek-V2-Lite widths (H=16, d_c=512, d_rope=64, d_nope=d_v=128)."""
    rng = np.random.default_rng(7)
    case = _rand_case(rng, B=1, H=16, d_c=512, d_rope=64, d_nope=128, d_v=128, S=64,
                      lengths=[64])
    case["w_uk"] *= 0.02 / 0.3
    case["w_uv"] *= 0.02 / 0.3
    a = O.decode_absorbed(**case, scale=192 ** -0.5, base=10000.0)
    n = O.decode_naive(**case, scale=192 ** -0.5, base=10000.0)
    assert np.max(np.abs(a["o"] - n["o"])) <= 1e-10


# ---------------------------------------------------------------- O-I2: softmax rows
def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(3)
    case = _rand_case(rng, S=31)
    a = O.decode_absorbed(**case, scale=0.3, base=10000.0)
    for b, p in enumerate(a["p"]):
        assert p.shape[1] == case["lengths"][b]
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12


# ---------------------------------------------------------------- O-I3: brute force
def _brute(q_nope, q_rope, w_uk, w_uv, cache, n, pos, scale, base):
    """Scalar loops over one sequence, written from the definitions directly."""
    H, d_nope = len(q_nope), len(q_nope[0])
    d_c = len(w_uk[0][0])
    d_rope = len(q_rope[0])
    d_v = len(w_uv[0])
    out_o, out_oc, out_lse = [], [], []
    for h in range(H):
        # absorbed query: contraction of q_nope with W_UK over d_nope
        qa = [sum(q_nope[h][d] * w_uk[h][d][c] for d in range(d_nope)) for c in range(d_c)]
        # rotate adjacent pairs by pos * base^(-2i/d_rope)
        qp = [0.0] * d_rope
        for i in range(d_rope // 2):
            ang = pos * base ** (-(2.0 * i) / d_rope)
            x0, x1 = q_rope[h][2 * i], q_rope[h][2 * i + 1]
            qp[2 * i] = math.cos(ang) * x0 - math.sin(ang) * x1
            qp[2 * i + 1] = math.sin(ang) * x0 + math.cos(ang) * x1
        s = []
        for t in range(n):
            v = sum(qa[c] * cache[t][c] for c in range(d_c))
            v += sum(qp[r] * cache[t][d_c + r] for r in range(d_rope))
            s.append(scale * v)
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        oc = [sum(e[t] / z * cache[t][c] for t in range(n)) for c in range(d_c)]
        o = [sum(w_uv[h][k][c] * oc[c] for c in range(d_c)) for k in range(d_v)]
        out_o.append(o)
        out_oc.append(oc)
        out_lse.append(m + math.log(z))
    return np.array(out_o), np.array(out_oc), np.array(out_lse)


@pytest.mark.parametrize("d_rope", [2, 4])
@pytest.mark.parametrize("H", [1, 2])
@pytest.mark.parametrize("S", [1, 2, 3])
def test_brute_force_tiny(H, S, d_rope):
    """With d_rope = 4 two frequencies meet two pairs, so the brute force also
    sees which frequency rotates which pair."""
    rng = np.random.default_rng(100 + 10 * H + S + 1000 * d_rope)
    case = _rand_case(rng, B=1, H=H, d_c=4, d_rope=d_rope, d_nope=2, d_v=3, S=S, lengths=[S])
    case["positions"] = np.array([5])
    scale = 0.5
    a = O.decode_absorbed(**case, scale=scale, base=10000.0)
    n = O.decode_naive(**case, scale=scale, base=10000.0)
    bo, boc, blse = _brute(case["q_nope"][0].tolist(), case["q_rope"][0].tolist(),
                           case["w_uk"].tolist(), case["w_uv"].tolist(),
                           case["cache"][0].tolist(), S, 5, scale, 10000.0)
    np.testing.assert_allclose(a["o"][0], bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(n["o"][0], bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(a["o_c"][0], boc, rtol=0, atol=1e-13)
    np.testing.assert_allclose(a["lse"][0], blse, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- O-I4: special cases
def test_single_row_returns_that_row():
    rng = np.random.default_rng(11)
    case = _rand_case(rng, B=1, lengths=[1])
    a = O.decode_absorbed(**case, scale=0.4, base=10000.0)
    row = case["cache"][0, 0, :16]
    for h in range(3):
        np.testing.assert_allclose(a["o_c"][0, h], row, atol=1e-15)
        np.testing.assert_allclose(a["o"][0, h], case["w_uv"][h] @ row, atol=1e-13)


def test_equal_rows_give_that_row_for_any_query():
    rng = np.random.default_rng(12)
    case = _rand_case(rng, B=1, S=6, lengths=[6])
    case["cache"][0, :, :] = case["cache"][0, 2, :]
    a = O.decode_absorbed(**case, scale=0.4, base=10000.0)
    assert np.max(np.abs(a["o_c"][0] - case["cache"][0, 0, :16][None])) <= 1e-14
    assert np.max(np.abs(a["p"][0] - 1.0 / 6)) <= 1e-14


def test_two_rows_logistic():
    """S=2: p_1 = sigma(s_1 - s_2), with the scores formed by hand."""
    rng = np.random.default_rng(13)
    case = _rand_case(rng, B=1, H=1, d_c=3, d_rope=2, d_nope=2, d_v=2, S=2, lengths=[2])
    case["positions"] = np.array([0])                  # RoPE is the identity at 0
    qn, qr = case["q_nope"][0, 0], case["q_rope"][0, 0]
    W = case["w_uk"][0]
    c = case["cache"][0]
    s = []
    for t in range(2):
        s.append(0.7 * (sum(qn[d] * W[d, k] * c[t, k] for d in range(2) for k in range(3))
                        + qr[0] * c[t, 3] + qr[1] * c[t, 4]))
    a = O.decode_absorbed(**case, scale=0.7, base=10000.0)
    p0 = 1.0 / (1.0 + math.exp(-(s[0] - s[1])))
    assert abs(a["p"][0][0, 0] - p0) <= 1e-14


def test_rope_identity_at_position_zero():
    x = np.random.default_rng(14).standard_normal((5, 64))
    np.testing.assert_array_equal(O.apply_rope(x, 0, 10000.0), x)


def test_rope_preserves_pair_norms():
    x = np.random.default_rng(15).standard_normal((7, 64))
    y = O.apply_rope(x, 12345, 10000.0)
    nx = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    ny = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-13)


def test_rope_width_two_is_plane_rotation():
    """With d_rope=2 the only frequency is base^0 = 1: a counter-clockwise rotation
    by `pos` radians, R = [[cos, -sin], [sin, cos]]."""
    for pos in [1, 3, 63, 4095]:
        x = np.array([0.3, -1.7])
        R = np.array([[math.cos(pos), -math.sin(pos)], [math.sin(pos), math.cos(pos)]])
        np.testing.assert_allclose(O.apply_rope(x, pos, 10000.0), R @ x, atol=1e-15)


def _rope_scalar(x, pos, base):
    """RoPE by scalar loops: pair i = (x[2i], x[2i+1]) is the complex number
    x[2i] + i x[2i+1] turned by the angle pos * base^(-2i/d) (Multi-Head Latent
    Attention, 3.7: frequencies from the even indices 0, 2, ..., d-2 over d, and
    the vector read as consecutive complex pairs in order)."""
    d = len(x)
    out = [0.0] * d
    for i in range(d // 2):
        ang = pos * base ** (-(2.0 * i) / d)
        out[2 * i] = math.cos(ang) * x[2 * i] - math.sin(ang) * x[2 * i + 1]
        out[2 * i + 1] = math.sin(ang) * x[2 * i] + math.cos(ang) * x[2 * i + 1]
    return np.array(out)


@pytest.mark.parametrize("d_rope,pos,base", [(6, 7, 10000.0), (8, 3, 10000.0),
                                             (64, 4095, 10000.0), (10, 11, 50.0)])
def test_rope_brute_force_pair_frequencies(d_rope, pos, base):
    """Several pairs at a position other than 0: every pair turns by its own
    frequency, so a frequency given to the wrong pair shows."""
    x = np.random.default_rng(17 + d_rope).standard_normal((3, d_rope))
    got = O.apply_rope(x, pos, base)
    for r in range(3):
        np.testing.assert_allclose(got[r], _rope_scalar(x[r].tolist(), pos, base),
                                   rtol=0, atol=1e-12)


def test_rope_each_pair_turns_by_its_own_angle():
    """A vector with a single nonzero pair i = (1, 0) comes back as
    (cos a, sin a) with a = pos * base^(-2i/d): the angle of pair i alone."""
    d, pos, base = 8, 3, 100.0
    for i in range(d // 2):
        x = np.zeros(d)
        x[2 * i] = 1.0
        y = O.apply_rope(x, pos, base)
        a = pos * base ** (-2.0 * i / d)       # 3, 0.95, 0.3, 0.095 radians
        assert abs(math.atan2(y[2 * i + 1], y[2 * i]) - a) <= 1e-14
        assert np.count_nonzero(np.delete(y, [2 * i, 2 * i + 1])) == 0


def test_rope_frequencies_closed_form():
    th = O.rope_theta(64, 10000.0)
    assert th[0] == 1.0
    assert abs(th[1] - 10000.0 ** (-1 / 32)) <= 2e-16          # within 1 ulp
    assert abs(th[-1] / 1e-4 ** (62 / 64) - 1) <= 4e-16
    assert np.all(np.diff(th) < 0)


def test_rope_relative_position():
    """<R_m q, R_n k> depends on m - n only (Multi-Head Latent Attention, eq. 3.4.2:
    R_i^T R_j is the rotation by the position difference)."""
    rng = np.random.default_rng(16)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    ref = O.apply_rope(q, 40, 10000.0) @ O.apply_rope(k, 17, 10000.0)
    for shift in [1, 100, 5000]:
        v = O.apply_rope(q, 40 + shift, 10000.0) @ O.apply_rope(k, 17 + shift, 10000.0)
        assert abs(v - ref) <= 1e-11 * (1 + abs(ref))


# ---------------------------------------------------------------- O-I5: KV-cache exactness
def test_decode_equals_last_row_of_causal_attention():
    """Decoding with the cache gives exactly the last row of full causal attention
    (Multi-Head Latent Attention, 2.1; "Transformer and KV Cache Basics", item 4)."""
    rng = np.random.default_rng(21)
    S, H, d_c, d_rope, d_nope, d_v = 11, 3, 16, 4, 6, 5
    qn = rng.standard_normal((S, H, d_nope))
    qr = rng.standard_normal((S, H, d_rope))
    c = rng.standard_normal((S, d_c))
    kr_raw = rng.standard_normal((S, d_rope))
    w_uk = 0.3 * rng.standard_normal((H, d_nope, d_c))
    w_uv = 0.3 * rng.standard_normal((H, d_v, d_c))
    kr = O.apply_rope(kr_raw, np.arange(S), 10000.0)       # keys rotated at their positions
    cache = np.concatenate([c, kr], axis=1)
    full = O.causal_attention_naive(qn, qr, w_uk, w_uv, cache, 0.3, 10000.0)
    for n in [1, 5, S]:                                   # decode at every cache length
        dec = O.decode_absorbed(qn[n - 1][None], qr[n - 1][None], w_uk, w_uv, cache[None],
                                np.array([n]), np.array([n - 1]), 0.3, 10000.0)
        np.testing.assert_allclose(dec["o"][0], full[n - 1], atol=1e-12)


# ---------------------------------------------------------------- O-I6: page counts
def test_op_counts_match_printed_totals():
    g = json.load(open(os.path.join(GOLDEN, "p2_op_counts.json")))
    dims = g["dims"]
    pr, ex = g["printed"], g["printed_expression_sums"]
    A = C.affine("A", **dims)
    assert A["flops"] == tuple(pr["A"]["flops"]) and A["memops"] == tuple(pr["A"]["memops"])
    B = C.affine("B", **dims)
    assert B["flops"] == tuple(pr["B"]["flops"])
    assert B["memops"][0] == pr["B"]["memops"][0]
    assert B["memops"] == tuple(ex["B"]["memops"])           # the page's terms, not its slip
    assert B["memops"][1] != pr["B"]["memops"][1]
    Cc = C.affine("C", **dims)
    assert Cc["flops"] == tuple(pr["C"]["flops"])
    assert Cc["memops"] == tuple(ex["C"]["memops"])
    assert Cc["memops"][1] != pr["C"]["memops"][1]
    # the materialised W_UK.W_Q pre-computation printed on the page
    assert dims["heads"] * dims["d_nope"] * dims["hidden"] * dims["d_c"] == pr["B"]["precompute_flops"]


def test_latent_path_counts():
    """The fully absorbed step touches each cached row once: 576 elements per row,
    H*(576+512) multiply-adds per row, constants from W_UK and W_UV."""
    a = C.affine("latent", heads=16)
    assert a["flops"] == (2 * 16 * 128 * 512, 16 * (576 + 512))
    assert a["memops"][1] == 576 + 512 + 2 * 16


def test_mla_over_mha_ratio():
    g = json.load(open(os.path.join(GOLDEN, "p1_ops_ratio.json")))
    v3 = g["v3"]
    r = v3["d_h"] * v3["H"] / v3["d_c"]
    assert r == v3["r"]
    ratio = C.mla_over_mha_ops(v3["d_h"], v3["H"], v3["d_c"], v3["d_h"] * v3["H"])
    assert abs(ratio - 3 / (2 * r)) < 1e-15
    assert 20 <= 1 / ratio < 22                                # "20x" printed; exact 21.33
    assert abs(C.mla_over_mha_ops(1, 3, 2, 3) - 1.0) < 1e-15  # r = 1.5 breaks even


# ---------------------------------------------------------------- O-I7: split + combine
@pytest.mark.parametrize("splits", [1, 2, 7, 128])
def test_split_combine_equals_unsplit(splits):
    rng = np.random.default_rng(30 + splits)
    S = 300
    case = _rand_case(rng, B=1, H=4, d_c=16, d_rope=4, d_nope=6, d_v=5, S=S, lengths=[S])
    case["cache"][0, ::37] *= 8.0                      # a few large rows, as in the long workload
    a = O.decode_absorbed(**case, scale=0.9, base=10000.0)
    chunk = -(-S // splits)
    oc, lse = O.split_decode_combine(a["q_abs"][0], a["q_pe"][0], case["cache"][0], S, 0.9, chunk)
    assert np.max(np.abs(oc - a["o_c"][0])) <= 1e-12
    assert np.max(np.abs(lse - a["lse"][0])) <= 1e-12


# ---------------------------------------------------------------- the pins catch planted mistakes
def test_pins_catch_a_transposed_operand(monkeypatch):
    """Plant W_UK^T (square dims) in the absorbed form: O-I1 must fail."""
    rng = np.random.default_rng(40)
    case = _rand_case(rng, B=1, H=2, d_c=6, d_rope=2, d_nope=6, d_v=3, S=5, lengths=[5])
    good = O.decode_naive(**case, scale=0.5, base=10000.0)["o"]
    monkeypatch.setattr(O, "absorb_q", lambda q, w: np.einsum("bhd,hcd->bhc", q, w))
    bad = O.decode_absorbed(**case, scale=0.5, base=10000.0)["o"]
    assert np.max(np.abs(bad - good)) > 1e-3


def test_pins_catch_a_wrong_rope_sign(monkeypatch):
    """Plant a clockwise rotation: the plane-rotation pin must fail."""
    orig = O.rope_theta
    monkeypatch.setattr(O, "rope_theta", lambda d, b: -orig(d, b))
    x = np.array([0.3, -1.7])
    R = np.array([[math.cos(3), -math.sin(3)], [math.sin(3), math.cos(3)]])
    assert np.max(np.abs(O.apply_rope(x, 3, 10000.0) - R @ x)) > 1e-3


def test_pins_catch_reversed_rope_frequencies(monkeypatch):
    """Plant the frequencies in reverse pair order (pair 0 turning slowest): the
    scalar RoPE pin and the d_rope = 4 brute force must both fail."""
    orig = O.rope_theta
    monkeypatch.setattr(O, "rope_theta", lambda d, b: orig(d, b)[::-1].copy())
    x = np.random.default_rng(23).standard_normal(6)
    assert np.max(np.abs(O.apply_rope(x, 7, 10000.0) - _rope_scalar(x.tolist(), 7, 10000.0))) > 1e-3
    rng = np.random.default_rng(100 + 10 * 2 + 3 + 4000)
    case = _rand_case(rng, B=1, H=2, d_c=4, d_rope=4, d_nope=2, d_v=3, S=3, lengths=[3])
    case["positions"] = np.array([5])
    bo, _, _ = _brute(case["q_nope"][0].tolist(), case["q_rope"][0].tolist(),
                      case["w_uk"].tolist(), case["w_uv"].tolist(),
                      case["cache"][0].tolist(), 3, 5, 0.5, 10000.0)
    bad = O.decode_absorbed(**case, scale=0.5, base=10000.0)["o"][0]
    assert np.max(np.abs(bad - bo)) > 1e-6


def test_pins_catch_a_dropped_rope_term(monkeypatch):
    """Plant a score without the k_rope part: brute force must disagree."""
    rng = np.random.default_rng(41)
    case = _rand_case(rng, B=1, H=1, d_c=4, d_rope=2, d_nope=2, d_v=3, S=3, lengths=[3])
    case["positions"] = np.array([5])
    bo, _, _ = _brute(case["q_nope"][0].tolist(), case["q_rope"][0].tolist(),
                      case["w_uk"].tolist(), case["w_uv"].tolist(),
                      case["cache"][0].tolist(), 3, 5, 0.5, 10000.0)
    mutated = dict(case)
    mutated["cache"] = case["cache"].copy()
    mutated["cache"][..., 4:] = 0.0
    bad = O.decode_absorbed(**mutated, scale=0.5, base=10000.0)["o"][0]
    assert np.max(np.abs(bad - bo)) > 1e-6


# ---------------------------------------------------------------- around the path
def test_cache_append_brute_force_tiny():
    """Scalar loops written out: y = W x, the last pair rotated by pos * theta."""
    rng = np.random.default_rng(3)
    d_c, d_r, hid = 3, 2, 4
    x = rng.standard_normal((2, hid))
    w = rng.standard_normal((d_c + d_r, hid))
    pos = np.array([0, 5])
    got = O.cache_append_row(x, w, pos, d_c, 10000.0)
    for b in range(2):
        y = [sum(w[o][k] * x[b][k] for k in range(hid)) for o in range(d_c + d_r)]
        for o in range(d_c):
            assert got[b, o] == pytest.approx(y[o], abs=1e-12)
        ang = pos[b] * 1.0          # theta_0 = base^0 = 1 for a single pair
        c, s = math.cos(ang), math.sin(ang)
        assert got[b, d_c] == pytest.approx(c * y[d_c] - s * y[d_c + 1], abs=1e-12)
        assert got[b, d_c + 1] == pytest.approx(s * y[d_c] + c * y[d_c + 1], abs=1e-12)


def test_appended_keys_give_relative_scores():
    """Keys appended at positions m and query rotated at position n score by n - m
    only: shifting every position by the same amount leaves all scores unchanged."""
    rng = np.random.default_rng(4)
    d_c, d_r, hid = 4, 8, 6
    w = rng.standard_normal((d_c + d_r, hid))
    xs = rng.standard_normal((5, hid))
    q = rng.standard_normal(d_r)
    def scores(shift):
        rows = np.stack([O.cache_append_row(xs[t:t + 1], w, [t + shift], d_c, 10000.0)[0]
                         for t in range(5)])
        qr = O.apply_rope(q, 4 + shift, 10000.0)
        return rows[:, d_c:] @ qr
    np.testing.assert_allclose(scores(0), scores(1234), rtol=0, atol=1e-9)


def test_output_projection_brute_force_and_identity():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((2, 3, 2))
    w = rng.standard_normal((4, 6))
    got = O.output_projection(o, w)
    for b in range(2):
        flat = [o[b, h, e] for h in range(3) for e in range(2)]
        for n in range(4):
            assert got[b, n] == pytest.approx(sum(w[n][k] * flat[k] for k in range(6)), abs=1e-12)
    np.testing.assert_allclose(O.output_projection(o, np.eye(6)), o.reshape(2, 6), atol=0)


# ----------------------------------------------------------------------------- FP8 E4M3 elements
def test_e4m3_decode_matches_library_and_format_landmarks():
    """Every one of the 256 codes decodes as torch's float8_e4m3fn does (a library
    routine); the format's landmark values hold (1.0, the largest 448, the
    smallest normal 2^-6 and subnormal 2^-9, the NaN patterns, signed zero)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256)
    mine = O.e4m3_to_float64(codes)
    lib = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    assert np.array_equal(mine[~np.isnan(mine)], lib[~np.isnan(lib)])
    v = O.e4m3_to_float64
    assert v(0x38) == 1.0 and v(0xB8) == -1.0
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert v(0x08) == 2.0 ** -6 and v(0x01) == 2.0 ** -9 and v(0x07) == 7 * 2.0 ** -9
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and np.signbit(v(0x80))
    assert int(np.isnan(mine).sum()) == 2


def test_e4m3_values_are_ordered_and_symmetric():
    """Sign-magnitude order: codes 0..126 increase strictly, code c + 128 is -value(c)."""
    pos = O.e4m3_to_float64(np.arange(127))
    assert np.all(np.diff(pos) > 0)
    neg = O.e4m3_to_float64(np.arange(128, 255))
    np.testing.assert_array_equal(neg, -pos)


def test_e4m3_round_is_nearest_even_and_saturating():
    """Round trip of every finite code; nearest-value rounding agrees with torch's
    float -> float8_e4m3fn conversion on values across the whole range; exact
    midpoints go to the even code; magnitudes past 448 saturate."""
    torch = pytest.importorskip("torch")
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(O.e4m3_round(O.e4m3_to_float64(codes)), codes)
    rng = np.random.default_rng(8)
    x = rng.standard_normal(3000) * np.exp2(rng.uniform(-11, 8, 3000))
    x = np.clip(x, -448.0, 448.0).astype(np.float32).astype(np.float64)
    lib = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_round(x), lib)
    # 1 + 1/16 lies halfway between 1 (0x38, even) and 1.125 (0x39)
    assert O.e4m3_round(1.0625) == 0x38 and O.e4m3_round(1.1875) == 0x3A
    assert O.e4m3_round(1e6) == 0x7E and O.e4m3_round(-1e6) == 0xFE


# ----------------------------------------------------------------------------- multi-token decode
def test_multi_token_decode_is_the_last_rows_of_causal_attention():
    """q_len new tokens decoded together give exactly the last q_len rows of full
    causal self-attention over the sequence ("Transformer and KV Cache Basics",
    Thinking item 4: only the small upper-right triangle is masked), for every
    q_len up to the whole sequence, through the naive (decompressed K/V) form."""
    rng = np.random.default_rng(23)
    S, H, d_c, d_rope, d_nope, d_v = 9, 2, 12, 4, 6, 5
    qn = rng.standard_normal((S, H, d_nope))
    qr = rng.standard_normal((S, H, d_rope))
    c = rng.standard_normal((S, d_c))
    kr = O.apply_rope(rng.standard_normal((S, d_rope)), np.arange(S), 10000.0)
    w_uk = 0.3 * rng.standard_normal((H, d_nope, d_c))
    w_uv = 0.3 * rng.standard_normal((H, d_v, d_c))
    cache = np.concatenate([c, kr], axis=1)
    full = O.causal_attention_naive(qn, qr, w_uk, w_uv, cache, 0.3, 10000.0)
    for T in (1, 2, 4, S):
        got = O.decode_multi_token(qn[S - T:][None], qr[S - T:][None], w_uk, w_uv, cache[None],
                                   np.array([S]), T, 0.3, 10000.0)
        np.testing.assert_allclose(got["o"][0], full[S - T:], atol=1e-12)


def test_multi_token_decode_reduces_to_single_token_decode():
    """Token i of the block equals a single-token decode at cache length
    k_len - q_len + i + 1 (its own position), per call output; with q_len = 1 the
    two functions agree on every output."""
    rng = np.random.default_rng(24)
    a = _rand_case(rng, B=2, H=3, S=10, lengths=[10, 7])
    T = 3
    qn = rng.standard_normal((2, T, 3, a["q_nope"].shape[-1]))
    qr = rng.standard_normal((2, T, 3, a["q_rope"].shape[-1]))
    got = O.decode_multi_token(qn, qr, a["w_uk"], a["w_uv"], a["cache"], a["lengths"], T,
                               0.4, 10000.0)
    for b in range(2):
        for i in range(T):
            n = int(a["lengths"][b]) - T + i + 1
            one = O.decode_absorbed(qn[b, i][None], qr[b, i][None], a["w_uk"], a["w_uv"],
                                    a["cache"][b:b + 1], np.array([n]), np.array([n - 1]),
                                    0.4, 10000.0)
            for k in ("q_abs", "q_pe", "o_c", "lse", "o"):
                np.testing.assert_allclose(got[k][b, i], one[k][0], atol=1e-12)


# ---------------------------------------------------------------- materialised W^KQ and W^OV
def _materialized_case(rng, B=2, H=3, d_c=6, d_rope=4, d_nope=4, d_v=5, d_in=7, d_out=9, S=6):
    a = _rand_case(rng, B=B, H=H, d_c=d_c, d_rope=d_rope, d_nope=d_nope, d_v=d_v, S=S)
    a["x"] = rng.standard_normal((B, d_in))
    a["w_q_nope"] = 0.4 * rng.standard_normal((H, d_nope, d_in))
    a["w_o"] = 0.4 * rng.standard_normal((d_out, H * d_v))
    # the query's nope part as the model computes it: one d_nope block per head
    a["q_nope"] = np.einsum("hdi,bi->bhd", a["w_q_nope"], a["x"])
    return a


def test_materialized_weights_brute_force_tiny():
    """W^KQ[h, c, i] = sum_d W^UK[h, d, c] W^UQ[h, d, i] and
    W^OV[n, h d_c + c] = sum_e W^O[n, h d_v + e] W^UV[h, e, c], by scalar loops
    ("Multi-Head Latent Attention", 3.3 and eq. 3.3.3)."""
    rng = np.random.default_rng(31)
    H, d_nope, d_c, d_in, d_v, d_out = 2, 3, 4, 5, 3, 4
    w_q = rng.standard_normal((H, d_nope, d_in))
    w_uk = rng.standard_normal((H, d_nope, d_c))
    w_o = rng.standard_normal((d_out, H * d_v))
    w_uv = rng.standard_normal((H, d_v, d_c))
    kq = O.materialize_wkq(w_q, w_uk)
    ov = O.materialize_wov(w_o, w_uv)
    assert kq.shape == (H, d_c, d_in) and ov.shape == (d_out, H * d_c)
    for h in range(H):
        for c in range(d_c):
            for i in range(d_in):
                v = 0.0
                for d in range(d_nope):
                    v += w_uk[h, d, c] * w_q[h, d, i]
                assert abs(kq[h, c, i] - v) < 1e-12
    for n in range(d_out):
        for h in range(H):
            for c in range(d_c):
                v = 0.0
                for e in range(d_v):
                    v += w_o[n, h * d_v + e] * w_uv[h, e, c]
                assert abs(ov[n, h * d_c + c] - v) < 1e-12


@pytest.mark.parametrize("seed", [0, 1])
def test_materialized_equals_absorbed_and_naive(seed):
    """The materialised form (W^KQ x, then W^OV on the latent outputs) gives the
    absorbed form's q_abs, o_c and lse, and W^O applied to the naive form's head
    outputs, to 1e-10: the absorption is associativity ("Multi-Head Latent
    Attention", 3.3 and eq. 3.3.3)."""
    rng = np.random.default_rng(40 + seed)
    a = _materialized_case(rng)
    ab = O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                           a["lengths"], a["positions"], 0.37, 10000.0)
    nv = O.decode_naive(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                        a["lengths"], a["positions"], 0.37, 10000.0)
    m = O.decode_materialized(a["x"], a["q_rope"], O.materialize_wkq(a["w_q_nope"], a["w_uk"]),
                              O.materialize_wov(a["w_o"], a["w_uv"]), a["cache"], a["lengths"],
                              a["positions"], 0.37, 10000.0)
    for k in ("q_abs", "q_pe", "o_c", "lse"):
        np.testing.assert_allclose(m[k], ab[k], atol=1e-10)
    np.testing.assert_allclose(m["y"], O.output_projection(nv["o"], a["w_o"]), atol=1e-10)


def test_pins_catch_a_misplaced_wov_block(monkeypatch):
    """A W^OV whose head blocks are taken from the wrong head fails the pin above."""
    real = O.materialize_wov

    def wrong(w_o, w_uv):
        return real(w_o, np.asarray(w_uv)[::-1])
    rng = np.random.default_rng(44)
    a = _materialized_case(rng)
    monkeypatch.setattr(O, "materialize_wov", wrong)
    nv = O.decode_naive(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                        a["lengths"], a["positions"], 0.37, 10000.0)
    m = O.decode_materialized(a["x"], a["q_rope"], O.materialize_wkq(a["w_q_nope"], a["w_uk"]),
                              O.materialize_wov(a["w_o"], a["w_uv"]), a["cache"], a["lengths"],
                              a["positions"], 0.37, 10000.0)
    assert np.max(np.abs(m["y"] - O.output_projection(nv["o"], a["w_o"]))) > 1e-3
