"""Pins of the fp64 oracle against what the mathematics fixes (CPU only).

HeyGen, "Avatar inference at scale" prints no worked values for the step, so
each oracle function is pinned by closed forms, invariants, an independent
complex-number formulation, exact rationals, and literal loops (tests/_brute.py)
on tiny shapes.  ``test_planted_*`` plant a mistake in a copy of an oracle
function and check that a pin catches it.
"""
import fractions
import math

import numpy as np
import pytest

import oracle as O
from tests import _brute

RNG = np.random.default_rng(1234)


def rand(*shape):
    return RNG.standard_normal(shape)


# ----------------------------------------------------------------- pins ----

def pin_softmax(softmax=O.softmax_rows):
    s = rand(7, 33) * 5
    p = softmax(s)
    assert np.all(p > 0)
    assert np.max(np.abs(p.sum(axis=-1) - 1.0)) < 1e-12
    # ratios of probabilities are exp of score differences
    r = p[:, 3] / p[:, 10]
    assert np.allclose(r, np.exp(s[:, 3] - s[:, 10]), rtol=1e-12, atol=0)


def pin_attention_closed_forms(attention=O.attention):
    B, Nq, H, D = 2, 5, 3, 16
    q = rand(B, Nq, H, D)
    v = rand(B, 9, H, D)
    k = rand(B, 9, H, D)
    # one key: O = V
    o = attention(q, [(k[:, :1], v[:, :1])])
    assert np.allclose(o, np.broadcast_to(v[:, :1], o.shape), atol=1e-13)
    # zero queries: O = mean(V)
    o = attention(np.zeros_like(q), [(k, v)])
    assert np.allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-13)
    # identical keys: O = mean(V)
    k_same = np.broadcast_to(k[:, :1], k.shape).copy()
    o = attention(q, [(k_same, v)])
    assert np.allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-13)
    # two keys, one query: O = sigmoid(s1 - s2) v1 + sigmoid(s2 - s1) v2
    q1 = rand(1, 1, 1, D)
    k2 = rand(1, 2, 1, D)
    v2 = rand(1, 2, 1, D)
    scale = 0.37
    o = attention(q1, [(k2, v2)], scale)[0, 0, 0]
    s1 = float(q1[0, 0, 0] @ k2[0, 0, 0]) * scale
    s2 = float(q1[0, 0, 0] @ k2[0, 1, 0]) * scale
    sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
    assert np.allclose(o, sig * v2[0, 0, 0] + (1 - sig) * v2[0, 1, 0], atol=1e-13)


def pin_attention_default_scale(attention=O.attention):
    # default scale is 1/sqrt(D): compare against the explicit value
    q, k, v = rand(1, 4, 2, 64), rand(1, 6, 2, 64), rand(1, 6, 2, 64)
    assert np.allclose(attention(q, [(k, v)]), attention(q, [(k, v)], 1.0 / 8.0), atol=1e-14)
    assert not np.allclose(attention(q, [(k, v)]), attention(q, [(k, v)], 1.0), atol=1e-3)


def pin_attention_invariances(attention=O.attention):
    B, Nq, H, D = 1, 6, 2, 8
    q = rand(B, Nq, H, D)
    k = rand(B, 20, H, D)
    v = rand(B, 20, H, D)
    base = attention(q, [(k, v)])
    perm = RNG.permutation(20)
    assert np.allclose(attention(q, [(k[:, perm], v[:, perm])]), base, atol=1e-13)
    # splitting the KV set into 2 or 3 segments, with an empty one, changes nothing
    assert np.allclose(attention(q, [(k[:, :7], v[:, :7]), (k[:, 7:], v[:, 7:])]), base, atol=1e-13)
    assert np.allclose(attention(q, [(k[:, :3], v[:, :3]), (k[:, 3:3], v[:, 3:3]), (k[:, 3:], v[:, 3:])]),
                       base, atol=1e-13)
    # heads and batches are independent
    q2 = q.copy()
    q2[:, :, 1] += 3.0
    o2 = attention(q2, [(k, v)])
    assert np.allclose(o2[:, :, 0], base[:, :, 0], atol=1e-14)
    assert not np.allclose(o2[:, :, 1], base[:, :, 1], atol=1e-3)


def pin_attention_large_scores(attention=O.attention):
    # scores scaled x50 stay finite and equal the naive formula (fp64 holds exp(~300))
    q, k, v = rand(1, 3, 1, 16), rand(1, 11, 1, 16), rand(1, 11, 1, 16)
    scale = 50.0 / 4.0
    o = attention(q, [(k, v)], scale)
    assert np.all(np.isfinite(o))
    s = np.einsum("nd,md->nm", q[0, :, 0], k[0, :, 0]) * scale
    assert s.max() < 700
    e = np.exp(s)
    naive = (e / e.sum(axis=1, keepdims=True)) @ v[0, :, 0]
    assert np.allclose(o[0, :, 0], naive, rtol=1e-12, atol=1e-12)


def pin_rope_complex(rope3d=O.rope3d):
    """Rotation = complex multiplication of a_j + i b_j by exp(i pos w_j)."""
    B, gt, gh, gw, H, D = 1, 3, 2, 5, 2, 64
    x = rand(B, gt * gh * gw, H, D)
    t0, base = -2, 10000.0
    out = rope3d(x, gt, gh, gw, t0, base)
    z = x[..., 0::2] + 1j * x[..., 1::2]
    p_t, p_h, p_w = 12, 10, 10  # D = 64: 32 pairs, a third (10) per spatial axis, 12 for time
    ang = np.zeros((gt * gh * gw, D // 2))
    n = 0
    for tt in range(gt):
        for hh in range(gh):
            for ww in range(gw):
                for j in range(p_t):
                    ang[n, j] = (t0 + tt) * base ** (-j / p_t)
                for j in range(p_h):
                    ang[n, p_t + j] = hh * base ** (-j / p_h)
                for j in range(p_w):
                    ang[n, p_t + p_h + j] = ww * base ** (-j / p_w)
                n += 1
    zr = z * np.exp(1j * ang)[None, :, None, :]
    assert np.allclose(out[..., 0::2], zr.real, atol=1e-12)
    assert np.allclose(out[..., 1::2], zr.imag, atol=1e-12)


def pin_rope_properties(rope3d=O.rope3d):
    D = 128
    assert sum(O.rope_axis_split(D)) == D // 2
    assert O.rope_axis_split(128) == (22, 21, 21)
    assert O.rope_axis_split(64) == (12, 10, 10)
    x = rand(2, 2 * 3 * 4, 3, D)
    out = rope3d(x, 2, 3, 4, 0, 10000.0)
    # pair norms preserved
    assert np.allclose(np.hypot(out[..., 0::2], out[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]),
                       atol=1e-12)
    # token 0 sits at (0, 0, 0): identity
    assert np.allclose(out[:, 0], x[:, 0], atol=1e-15)
    # a token at (0, 0, w) only turns the w pairs, pair 0 of the axis by w radians
    tok = 3  # (t, h, w) = (0, 0, 3)
    p_t, p_h, p_w = O.rope_axis_split(D)
    moved = ~np.isclose(out[:, tok], x[:, tok], atol=1e-14)
    pair_moved = moved[..., 0::2] | moved[..., 1::2]
    assert not pair_moved[..., : p_t + p_h].any()
    assert pair_moved[..., p_t + p_h:].all()
    za = x[0, tok, 0, 2 * (p_t + p_h)] + 1j * x[0, tok, 0, 2 * (p_t + p_h) + 1]
    zb = out[0, tok, 0, 2 * (p_t + p_h)] + 1j * out[0, tok, 0, 2 * (p_t + p_h) + 1]
    assert abs(np.angle(zb / za) - 3.0) < 1e-12
    # the middle pair of the t axis turns at base**-0.5 = 0.01 rad per frame
    y = rand(1, 2, 1, D)
    r = rope3d(y, 2, 1, 1, 0, 10000.0)  # token 1 at t = 1
    j = p_t // 2
    za = y[0, 1, 0, 2 * j] + 1j * y[0, 1, 0, 2 * j + 1]
    zb = r[0, 1, 0, 2 * j] + 1j * r[0, 1, 0, 2 * j + 1]
    assert abs(np.angle(zb / za) - 10000.0 ** (-j / p_t)) < 1e-12
    assert abs(10000.0 ** (-11 / 22) - 0.01) < 1e-15


def pin_rope_relative(rope3d=O.rope3d):
    """Scores depend only on position differences: shifting every t by c
    leaves q.k unchanged."""
    D, gt, gh, gw = 64, 3, 2, 3
    q = rand(1, gt * gh * gw, 1, D)
    k = rand(1, gt * gh * gw, 1, D)
    s0 = np.einsum("nd,md->nm", rope3d(q, gt, gh, gw, 0)[0, :, 0], rope3d(k, gt, gh, gw, 0)[0, :, 0])
    s1 = np.einsum("nd,md->nm", rope3d(q, gt, gh, gw, 17)[0, :, 0], rope3d(k, gt, gh, gw, 17)[0, :, 0])
    assert np.allclose(s0, s1, atol=1e-11)
    # ... and do depend on the difference
    s2 = np.einsum("nd,md->nm", rope3d(q, gt, gh, gw, 0)[0, :, 0], rope3d(k, gt, gh, gw, 5)[0, :, 0])
    assert not np.allclose(s0, s2, atol=1e-3)


def pin_out_proj_euler(out_proj=O.out_proj, euler=O.euler_update):
    sq = rand(12, 12)
    o = rand(5, 12)
    assert np.allclose(out_proj(o, sq), np.array(_brute.linear(o.tolist(), sq.tolist())), atol=1e-12)
    w, b, x = rand(7, 12), rand(7), rand(5, 7)
    ref = _brute.linear(o.tolist(), w.tolist(), b.tolist())
    assert np.allclose(out_proj(o, w, b), np.array(ref), atol=1e-12)
    ref_nb = _brute.linear(o.tolist(), w.tolist())
    assert np.allclose(out_proj(o, w), np.array(ref_nb), atol=1e-12)
    v = rand(5, 7)
    xe = euler(x, v, 0.25)
    assert np.allclose(xe - x, 0.25 * v, atol=1e-15)


def pin_time_grid(time_grid=O.time_grid):
    for S in (1, 4, 8, 30):
        u = time_grid(S, 1.0)
        assert np.allclose(u, 1.0 / S, atol=1e-15)
    for S, shift in ((30, 3.0), (8, 2.0), (30, 5.0)):
        dt = time_grid(S, shift)
        assert abs(dt.sum() - 1.0) < 1e-14 and np.all(dt > 0)
    # shift 3 over S steps: warped level of step i is 3(S-i)/(3S-2i) exactly
    S = 30
    lev = [fractions.Fraction(3 * (S - i), 3 * S - 2 * i) for i in range(S + 1)]
    exact = [float(lev[i] - lev[i + 1]) for i in range(S)]
    assert np.allclose(time_grid(S, 3.0), exact, rtol=1e-13, atol=0)
    assert abs(exact[0] - 1 / 88) < 1e-15 and abs(exact[-1] - 3 / 32) < 1e-15
    # a constant velocity integrates to x0 + v over any grid
    x0, v = rand(4, 3), rand(4, 3)
    x = x0.copy()
    for dt in time_grid(30, 3.0):
        x = O.euler_update(x, v, dt)
    assert np.allclose(x, x0 + v, atol=1e-13)


# ------------------------------------------------------------ the tests ----

def test_softmax_rows():
    pin_softmax()


def test_attention_closed_forms():
    pin_attention_closed_forms()


def test_attention_default_scale():
    pin_attention_default_scale()


def test_attention_invariances():
    pin_attention_invariances()


def test_attention_large_scores():
    pin_attention_large_scores()


def test_rope_complex():
    pin_rope_complex()


def test_rope_properties():
    pin_rope_properties()


def test_rope_relative():
    pin_rope_relative()


def test_out_proj_euler():
    pin_out_proj_euler()


def test_time_grid():
    pin_time_grid()


def _tiny_case(seed=7, n_b_frames=0):
    B, H, D, F, gh, gw = 1, 2, 64, 2, 4, 4
    N = F * gh * gw
    R = gh * gw
    Nb = n_b_frames * gh * gw
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((B, N, H, D)) for _ in range(3))
    rk, rv = rng.standard_normal((B, R, H, D)), rng.standard_normal((B, R, H, D))
    bk, bv = rng.standard_normal((B, Nb, H, D)), rng.standard_normal((B, Nb, H, D))
    w = rng.standard_normal((H * D, H * D)) / math.sqrt(H * D)
    x = rng.standard_normal((B * N, H * D))
    return dict(q=q, k=k, v=v, rk=rk, rv=rv, bk=bk, bv=bv, w=w, x=x, B=B, H=H, D=D, F=F, gh=gh, gw=gw,
                Tb=n_b_frames)


@pytest.mark.parametrize("tb", [0, 1])
def test_step_equals_brute_force(tb):
    c = _tiny_case(n_b_frames=tb)
    base, dt = 10000.0, 0.25
    rk_rot = O.rope3d(c["rk"], 1, c["gh"], c["gw"], -1, base)
    bk_rot = O.rope3d(c["bk"], tb, c["gh"], c["gw"], -tb, base) if tb else c["bk"]
    x1, o = O.chunk_step(c["q"], c["k"], c["v"], rk_rot, c["rv"], bk_rot, c["bv"], c["w"], c["x"], dt,
                         (c["F"], c["gh"], c["gw"]), base)
    # literal loops
    qr = _brute.rope_block(c["q"], c["F"], c["gh"], c["gw"], 0, base)[0]
    kr = _brute.rope_block(c["k"], c["F"], c["gh"], c["gw"], 0, base)[0]
    rkr = _brute.rope_block(c["rk"], 1, c["gh"], c["gw"], -1, base)[0]
    keys = rkr + kr
    vals = [[list(h) for h in tok] for tok in c["rv"][0]] + [[list(h) for h in tok] for tok in c["v"][0]]
    if tb:
        bkr = _brute.rope_block(c["bk"], tb, c["gh"], c["gw"], -tb, base)[0]
        keys = rkr + bkr + kr
        vals = ([[list(h) for h in tok] for tok in c["rv"][0]] + [[list(h) for h in tok] for tok in c["bv"][0]]
                + [[list(h) for h in tok] for tok in c["v"][0]])
    ob = _brute.attend(qr, keys, vals, 1.0 / math.sqrt(c["D"]))
    assert np.allclose(o[0], np.array(ob), atol=1e-12)
    flat = [[e for head in tok for e in head] for tok in ob]
    vel = _brute.linear(flat, c["w"].tolist())
    xb = c["x"] + dt * np.array(vel)
    assert np.allclose(x1, xb, atol=1e-12)


def test_chunk0_without_boundary_is_ref_plus_chunk():
    c = _tiny_case()
    rk_rot = O.rope3d(c["rk"], 1, c["gh"], c["gw"], -1)
    empty = np.zeros((1, 0, c["H"], c["D"]))
    qr = O.rope3d(c["q"], c["F"], c["gh"], c["gw"], 0)
    kr = O.rope3d(c["k"], c["F"], c["gh"], c["gw"], 0)
    a = O.attention(qr, [(rk_rot, c["rv"]), (empty, empty), (kr, c["v"])])
    b = O.attention(qr, [(np.concatenate([rk_rot, kr], 1), np.concatenate([c["rv"], c["v"]], 1))])
    assert np.allclose(a, b, atol=1e-13)


def test_stream_boundary_roll():
    """The boundary used by chunk c+1 is chunk c's last-step K/V tail, K
    re-rotated to t = -Tb..-1; chunk 0 equals a stand-alone step."""
    from streaming_avatar_video_gb300.inputs import Workload
    w = Workload("t", B=1, H=2, D=64, F=3, grid_h=2, grid_w=3, ref_frames=1, boundary_frames=2,
                 steps=2, shift=1.0, chunks=3)
    rng = np.random.default_rng(5)
    shp = (w.B, w.n_q, w.H, w.D)
    ins = {(c, s): tuple(rng.standard_normal(shp) for _ in range(3)) for c in range(3) for s in range(2)}
    x0 = {c: rng.standard_normal((w.B * w.n_q, w.hid)) for c in range(3)}
    rk, rv = rng.standard_normal((1, w.n_ref, w.H, w.D)), rng.standard_normal((1, w.n_ref, w.H, w.D))
    wo = rng.standard_normal((w.hid, w.hid)) / 8
    dts = O.time_grid(2, 1.0)
    xs, bnds = O.run_stream(w, rk, rv, wo, lambda c: x0[c], lambda c, s: ins[(c, s)], dts)
    assert bnds[0][0].shape[1] == 0
    for c in (1, 2):
        k_last, v_last = ins[(c - 1, 1)][1], ins[(c - 1, 1)][2]
        tail = k_last[:, w.n_q - w.n_b:]
        assert np.allclose(bnds[c][0], O.rope3d(tail, 2, w.grid_h, w.grid_w, -2), atol=1e-14)
        assert np.allclose(bnds[c][1], v_last[:, w.n_q - w.n_b:], atol=0)
        # the tail frames sat at t = F-2, F-1 of the finished chunk: same relative geometry
        full = O.rope3d(k_last, w.F, w.grid_h, w.grid_w, -w.F)
        assert np.allclose(bnds[c][0], full[:, w.n_q - w.n_b:], atol=1e-12)
    # chunk 0 by hand
    rk_rot = O.rope3d(rk, 1, w.grid_h, w.grid_w, -1)
    empty = np.zeros((1, 0, w.H, w.D))
    x = x0[0]
    for s, dt in enumerate(dts):
        x, _ = O.chunk_step(*ins[(0, s)], rk_rot, rv, empty, empty, wo, x, dt, (w.F, w.grid_h, w.grid_w))
    assert np.allclose(xs[0], x, atol=1e-13)


# ------------------------------------------- planted mistakes are caught ----

def _expect_pin_failure(pin, *mutated):
    with pytest.raises(AssertionError):
        pin(*mutated)


def test_planted_rope_sign():
    def bad(x, gt, gh, gw, t0=0, base=10000.0):
        # turns every pair the wrong way: conj(rope(conj(x)))
        y = x.copy()
        y[..., 1::2] *= -1
        r = O.rope3d(y, gt, gh, gw, t0, base)
        r[..., 1::2] *= -1
        return r
    _expect_pin_failure(pin_rope_complex, bad)


def test_planted_rope_axis_swap():
    def bad(x, gt, gh, gw, t0=0, base=10000.0):
        # h and w positions exchanged (only differs when gh != gw)
        B, N, H, D = x.shape
        y = x.reshape(B, gt, gh, gw, H, D).transpose(0, 1, 3, 2, 4, 5).reshape(B, N, H, D)
        r = O.rope3d(y, gt, gw, gh, t0, base)
        return r.reshape(B, gt, gw, gh, H, D).transpose(0, 1, 3, 2, 4, 5).reshape(B, N, H, D)
    # rotating with swapped grid gives (h' = w) positions: caught by the complex pin
    _expect_pin_failure(pin_rope_complex, bad)


def test_planted_rope_frequency():
    def bad(x, gt, gh, gw, t0=0, base=10000.0):
        return O.rope3d(x, gt, gh, gw, t0, base * 2)
    _expect_pin_failure(pin_rope_complex, bad)


def test_planted_attention_no_scale():
    def bad(q, segs, scale=None):
        return O.attention(q, segs, 1.0)
    _expect_pin_failure(pin_attention_default_scale, bad)


def test_planted_attention_k_for_v():
    def bad(q, segs, scale=None):
        return O.attention(q, [(k, k) for k, _ in segs], scale)
    _expect_pin_failure(pin_attention_closed_forms, bad)


def test_planted_attention_drops_segment():
    def bad(q, segs, scale=None):
        return O.attention(q, segs[:2] if len(segs) > 2 else segs, scale)
    _expect_pin_failure(pin_attention_invariances, bad)


def test_planted_softmax_no_normalise():
    def bad(s):
        return np.exp(s - s.max(axis=-1, keepdims=True))
    _expect_pin_failure(pin_softmax, bad)


def test_planted_out_proj_transpose():
    def bad(o, w, bias=None):
        v = o @ w if w.shape[0] == w.shape[1] else o @ w.T
        return v if bias is None else v + bias[None, :]
    _expect_pin_failure(pin_out_proj_euler, bad)


def test_planted_euler_sign():
    def bad(x, v, dt):
        return x - dt * v
    _expect_pin_failure(pin_out_proj_euler, O.out_proj, bad)


def test_planted_time_grid_off_by_one():
    def bad(steps, shift=1.0):
        sigma = 1.0 - np.arange(steps + 1, dtype=np.float64) / (steps + 1)
        warped = shift * sigma / (1.0 + (shift - 1.0) * sigma)
        return warped[:-1] - warped[1:]
    _expect_pin_failure(pin_time_grid, bad)


# ------------------------------------------------- interpolation chunks ----

def _i_case(seed=11, F=4, gh=2, gw=3, H=2, D=64):
    rng = np.random.default_rng(seed)
    ft = gh * gw
    n_int = (F - 2) * ft
    q, k, v = (rng.standard_normal((1, n_int, H, D)) for _ in range(3))
    ap = (rng.standard_normal((1, ft, H, D)), rng.standard_normal((1, ft, H, D)))
    an = (rng.standard_normal((1, ft, H, D)), rng.standard_normal((1, ft, H, D)))
    rk, rv = rng.standard_normal((1, ft, H, D)), rng.standard_normal((1, ft, H, D))
    w = rng.standard_normal((H * D, H * D)) / math.sqrt(H * D)
    x = rng.standard_normal((n_int, H * D))
    return dict(q=q, k=k, v=v, ap=ap, an=an, rk=rk, rv=rv, w=w, x=x, F=F, gh=gh, gw=gw, H=H, D=D)


def pin_ichunk_brute(ichunk=O.ichunk_step):
    """Literal loops: interior frames at t = 1..F-2, anchors at t = 0 and F-1."""
    c = _i_case()
    base, dt, F, gh, gw, D = 10000.0, 0.5, c["F"], c["gh"], c["gw"], c["D"]
    rk_rot = O.rope3d(c["rk"], 1, gh, gw, -1, base)
    x1, o = ichunk(c["q"], c["k"], c["v"], rk_rot, c["rv"], c["ap"], c["an"], c["w"], c["x"], dt, (F, gh, gw), base)
    qr = _brute.rope_block(c["q"], F - 2, gh, gw, 1, base)[0]
    keys = (_brute.rope_block(c["rk"], 1, gh, gw, -1, base)[0]
            + _brute.rope_block(c["ap"][0], 1, gh, gw, 0, base)[0]
            + _brute.rope_block(c["k"], F - 2, gh, gw, 1, base)[0]
            + _brute.rope_block(c["an"][0], 1, gh, gw, F - 1, base)[0])
    lst = lambda a: [[list(h) for h in tok] for tok in a[0]]
    vals = lst(c["rv"]) + lst(c["ap"][1]) + lst(c["v"]) + lst(c["an"][1])
    ob = _brute.attend(qr, keys, vals, 1.0 / math.sqrt(D))
    assert np.allclose(o[0], np.array(ob), atol=1e-12)
    flat = [[e for head in tok for e in head] for tok in ob]
    assert np.allclose(x1, c["x"] + dt * np.array(_brute.linear(flat, c["w"].tolist())), atol=1e-12)


def test_ichunk_equals_brute_force():
    pin_ichunk_brute()


def test_ichunk_relative_time():
    """Shifting the whole I chunk's time by one frame (anchors at -1 and F-2,
    interior from 0) changes nothing: its attention equals an N-style step
    whose two context frames sit at those times."""
    c = _i_case(seed=3)
    F, gh, gw = c["F"], c["gh"], c["gw"]
    empty = np.zeros((1, 0, c["H"], c["D"]))
    x1, o = O.ichunk_step(c["q"], c["k"], c["v"], empty, empty, c["ap"], c["an"], c["w"], c["x"], 0.5, (F, gh, gw))
    q_rot = O.rope3d(c["q"], F - 2, gh, gw, 0)
    k_rot = O.rope3d(c["k"], F - 2, gh, gw, 0)
    a0 = O.rope3d(c["ap"][0], 1, gh, gw, -1)
    a1 = O.rope3d(c["an"][0], 1, gh, gw, F - 2)
    o2 = O.attention(q_rot, [(a0, c["ap"][1]), (k_rot, c["v"]), (a1, c["an"][1])])
    assert np.allclose(o, o2, atol=1e-12)


def test_stream_ni_schedule_and_anchors():
    """I_k runs after N_{k+1}; its anchors are N_k's last frame and N_{k+1}'s
    first frame, both from their final steps."""
    from streaming_avatar_video_gb300.inputs import Workload
    w = Workload("ni", B=1, H=2, D=64, F=4, grid_h=2, grid_w=2, ref_frames=1, boundary_frames=1,
                 steps=2, shift=1.0)
    rng = np.random.default_rng(9)
    shp = (1, w.n_q, w.H, w.D)
    ishp = (1, (w.F - 2) * w.frame_tokens, w.H, w.D)
    n_in = {(c, s): tuple(rng.standard_normal(shp) for _ in range(3)) for c in range(3) for s in range(2)}
    i_in = {(c, s): tuple(rng.standard_normal(ishp) for _ in range(3)) for c in range(2) for s in range(2)}
    rk, rv = rng.standard_normal((1, w.n_ref, w.H, w.D)), rng.standard_normal((1, w.n_ref, w.H, w.D))
    wo = rng.standard_normal((w.hid, w.hid)) / 8
    xs_n, xs_i, used = O.run_stream_ni(
        w, rk, rv, wo, lambda c: np.zeros((w.n_q, w.hid)), lambda c: np.zeros((ishp[1], w.hid)),
        lambda c, s: n_in[(c, s)], lambda c, s: i_in[(c, s)], O.time_grid(2), O.time_grid(2), 3)
    assert len(xs_n) == 3 and len(xs_i) == 2
    ft = w.frame_tokens
    for k in range(2):
        a_prev, a_next = used[k]
        assert np.array_equal(a_prev[0], n_in[(k, 1)][1][:, w.n_q - ft:])
        assert np.array_equal(a_prev[1], n_in[(k, 1)][2][:, w.n_q - ft:])
        assert np.array_equal(a_next[0], n_in[(k + 1, 1)][1][:, :ft])
        assert np.array_equal(a_next[1], n_in[(k + 1, 1)][2][:, :ft])
    # the N chunks are unaffected by the I chunks: same as the plain stream
    xs_plain, _ = O.run_stream(w, rk, rv, wo, lambda c: np.zeros((w.n_q, w.hid)), lambda c, s: n_in[(c, s)],
                               O.time_grid(2), chunks=3)
    for c in range(3):
        assert np.allclose(xs_n[c], xs_plain[c], atol=0)


def test_planted_ichunk_anchor_times():
    # both anchors rotated to t = 0: the literal-loop pin must fail
    _expect_pin_failure(pin_ichunk_brute, _bad_ichunk)


def _bad_ichunk(q, k, v, rk, rv, ap, an, w_o, x, dt, grid, base=10000.0, scale=None, bias=None):
    F, gh, gw = grid
    q_rot = O.rope3d(q, F - 2, gh, gw, 1, base)
    k_rot = O.rope3d(k, F - 2, gh, gw, 1, base)
    a = np.concatenate([O.rope3d(ap[0], 1, gh, gw, 0, base), O.rope3d(an[0], 1, gh, gw, 0, base)], axis=1)
    o = O.attention(q_rot, [(rk, rv), (a, np.concatenate([ap[1], an[1]], axis=1)), (k_rot, v)])
    B, Nq, H, D = o.shape
    return O.euler_update(x, O.out_proj(o.reshape(B * Nq, H * D), w_o), dt), o


# ---------------------------------------------------- DiT attention block ----

def pin_qkv_project(qkv=O.qkv_project):
    """The projection is a literal triple loop, split as [q | k | v] along the
    output features and reshaped head-major."""
    rng = np.random.default_rng(21)
    B, N, H, D = 2, 3, 2, 4
    hid = H * D
    x = rng.standard_normal((B * N, hid))
    w = rng.standard_normal((3 * hid, hid))
    q, k, v = qkv(x, w, B, H, D)
    full = np.array(_brute.linear(x.tolist(), w.tolist()))
    for i, t in enumerate((q, k, v)):
        assert t.shape == (B, N, H, D)
        assert np.allclose(t.reshape(B * N, hid), full[:, i * hid:(i + 1) * hid], atol=1e-12)
    assert np.allclose(q[1, 2, 1], full[5, 4:8], atol=1e-12)


def test_qkv_project():
    pin_qkv_project()


def test_planted_qkv_order():
    def bad(x, w, B, H, D):
        q, k, v = O.qkv_project(x, w, B, H, D)
        return k, q, v
    _expect_pin_failure(pin_qkv_project, bad)


def test_block_step_is_projection_then_chunk_step():
    rng = np.random.default_rng(4)
    B, H, D, F, gh, gw = 1, 2, 64, 2, 2, 3
    N, hid = F * gh * gw, H * D
    x = rng.standard_normal((B * N, hid))
    wq = rng.standard_normal((3 * hid, hid)) / math.sqrt(hid)
    wo = rng.standard_normal((hid, hid)) / math.sqrt(hid)
    rk, rv = rng.standard_normal((B, gh * gw, H, D)), rng.standard_normal((B, gh * gw, H, D))
    empty = np.zeros((B, 0, H, D))
    x1, k, v = O.block_step(x, wq, rk, rv, empty, empty, wo, 0.3, (F, gh, gw), H, D)
    qkv = np.array(_brute.linear(x.tolist(), wq.tolist()))
    q2 = qkv[:, :hid].reshape(B, N, H, D)
    k2 = qkv[:, hid:2 * hid].reshape(B, N, H, D)
    v2 = qkv[:, 2 * hid:].reshape(B, N, H, D)
    x2, _ = O.chunk_step(q2, k2, v2, rk, rv, empty, empty, wo, x, 0.3, (F, gh, gw))
    assert np.allclose(x1, x2, atol=1e-12)
    assert np.allclose(k, k2, atol=1e-12) and np.allclose(v, v2, atol=1e-12)


# ------------------------------------------ block stream (rolled boundary) ----

def _block_stream_case(seed=31):
    from streaming_avatar_video_gb300.inputs import Workload
    w = Workload("tb", B=1, H=2, D=8, F=2, grid_h=2, grid_w=2, ref_frames=1, boundary_frames=1,
                 steps=2, shift=1.0, chunks=3)
    rng = np.random.default_rng(seed)
    rk, rv = rng.standard_normal((1, w.n_ref, w.H, w.D)), rng.standard_normal((1, w.n_ref, w.H, w.D))
    wq = rng.standard_normal((3 * w.hid, w.hid)) / math.sqrt(w.hid)
    wo = rng.standard_normal((w.hid, w.hid)) / math.sqrt(w.hid)
    bias = rng.standard_normal(w.hid) / 4
    x0 = {c: rng.standard_normal((w.B * w.n_q, w.hid)) for c in range(3)}
    return w, rk, rv, wq, wo, bias, x0, [0.375, 0.625]


def _brute_block_stream(w, rk, rv, wq, wo, bias, x0, dts, chunks, base=10000.0):
    """The block stream written as literal loops: the state is projected to
    q, k, v by a triple loop, every head vector rotated pair by pair, attention
    by explicit sums over [reference | boundary | chunk], W_o by a triple loop
    and the Euler update element by element.  The boundary of chunk c+1 is the
    last frame of chunk c's keys and values as projected at its final step, the
    keys rotated to t = -1."""
    H, D, hid = w.H, w.D, w.hid
    ref_rot = _brute.rope_block(rk, w.ref_frames, w.grid_h, w.grid_w, w.ref_t - w.ref_frames + 1, base)[0]
    ref_v = [[list(map(float, hv)) for hv in tok] for tok in rv[0]]
    bnd_k, bnd_v = [], []
    xs, used = [], []
    for c in range(chunks):
        used.append((bnd_k, bnd_v))
        x = [list(map(float, r)) for r in x0[c]]
        for dt in dts:
            qkv = _brute.linear(x, wq.tolist())
            split = lambda i: [[r[i * hid + hh * D: i * hid + (hh + 1) * D] for hh in range(H)] for r in qkv]  # noqa: E731
            q, k, v = split(0), split(1), split(2)
            qr = _brute.rope_block([q], w.F, w.grid_h, w.grid_w, 0, base)[0]
            kr = _brute.rope_block([k], w.F, w.grid_h, w.grid_w, 0, base)[0]
            o = _brute.attend(qr, ref_rot + bnd_k + kr, ref_v + bnd_v + v, 1.0 / math.sqrt(D))
            vel = _brute.linear([[e for hv in tok for e in hv] for tok in o], wo.tolist(), bias.tolist())
            x = [[x[i][j] + dt * vel[i][j] for j in range(hid)] for i in range(len(x))]
        xs.append(np.array(x))
        tail = w.n_q - w.n_b
        bnd_k = _brute.rope_block([k[tail:]], w.boundary_frames, w.grid_h, w.grid_w, -w.boundary_frames, base)[0]
        bnd_v = [[list(hv) for hv in tok] for tok in v[tail:]]
    return xs, used


def pin_stream_block(run=O.run_stream_block):
    w, rk, rv, wq, wo, bias, x0, dts = _block_stream_case()
    xs, bnds = run(w, rk, rv, wq, wo, lambda c: x0[c], np.array(dts), 3, None, bias)
    want_x, want_b = _brute_block_stream(w, rk, rv, wq, wo, bias, x0, dts, 3)
    assert len(xs) == 3 and len(bnds) == 3
    assert bnds[0][0].shape[1] == 0
    for c in range(3):
        assert np.allclose(xs[c], want_x[c], atol=1e-12), f"chunk {c} x"
        if c > 0:
            assert np.allclose(bnds[c][0][0], np.array(want_b[c][0]), atol=1e-12), f"chunk {c} boundary k"
            assert np.allclose(bnds[c][1][0], np.array(want_b[c][1]), atol=1e-12), f"chunk {c} boundary v"


def test_stream_block_equals_brute_force():
    pin_stream_block()


def test_stream_block_boundary_is_last_step_tail():
    """Chunk c+1's boundary is the tail of chunk c's final-step projection:
    the k, v that block_step returns for the last dt, k rotated to -T_b..-1."""
    w, rk, rv, wq, wo, bias, x0, dts = _block_stream_case(seed=32)
    xs, bnds = O.run_stream_block(w, rk, rv, wq, wo, lambda c: x0[c], np.array(dts), 2, None, bias)
    rk_rot = O.rope3d(rk, 1, w.grid_h, w.grid_w, -1)
    empty = np.zeros((1, 0, w.H, w.D))
    x = x0[0]
    x, k0, v0 = O.block_step(x, wq, rk_rot, rv, empty, empty, wo, dts[0], (w.F, w.grid_h, w.grid_w), w.H, w.D,
                             bias=bias)
    x, k1, v1 = O.block_step(x, wq, rk_rot, rv, empty, empty, wo, dts[1], (w.F, w.grid_h, w.grid_w), w.H, w.D,
                             bias=bias)
    assert np.allclose(xs[0], x, atol=1e-13)
    tail = w.n_q - w.n_b
    assert np.allclose(bnds[1][0], O.rope3d(k1[:, tail:], 1, w.grid_h, w.grid_w, -1), atol=1e-14)
    assert np.array_equal(bnds[1][1], v1[:, tail:])
    # the first step's projection differs, so a roll from it would be caught
    assert not np.allclose(k0[:, tail:], k1[:, tail:], atol=1e-3)


def _planted_block_stream(first_step_boundary=False, ref_t_shift=0):
    def run(w, ref_k, ref_v, w_qkv, w_o, x0_per_chunk, dts, chunks, scale=None, bias=None):
        ref_k_rot = O.rope3d(ref_k, w.ref_frames, w.grid_h, w.grid_w,
                             w.ref_t - w.ref_frames + 1 + ref_t_shift, w.rope_base)
        empty = np.zeros((w.B, 0, w.H, w.D))
        bnd = (empty, empty)
        xs, bnds = [], []
        for c in range(chunks):
            x = x0_per_chunk(c)
            bnds.append(bnd)
            kv = None
            for dt in dts:
                x, k, v = O.block_step(x, w_qkv, ref_k_rot, ref_v, bnd[0], bnd[1], w_o, dt,
                                       (w.F, w.grid_h, w.grid_w), w.H, w.D, w.rope_base, scale, bias)
                if kv is None or not first_step_boundary:
                    kv = (k, v)
            xs.append(x)
            bnd = O.boundary_from_chunk(kv[0], kv[1], w.frame_tokens, w.boundary_frames, w.grid_h, w.grid_w,
                                        w.rope_base)
        return xs, bnds
    return run


def test_planted_block_stream_first_step_boundary():
    # the boundary rolled from the chunk's first step instead of its last
    _expect_pin_failure(pin_stream_block, _planted_block_stream(first_step_boundary=True))


def test_planted_block_stream_reference_time():
    # the reference rotated at t = 0 instead of t = -1
    _expect_pin_failure(pin_stream_block, _planted_block_stream(ref_t_shift=1))


def test_planted_block_stream_control():
    # the planted copy with no mistake passes the pin (the two above fail for their mistake alone)
    pin_stream_block(_planted_block_stream())
